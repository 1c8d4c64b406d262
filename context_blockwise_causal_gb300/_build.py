"""Build step for libcpattn.so (the C-ABI library), in-tree, for sm_103a,
and for libcpattn_checked.so, the same library with the kernels' bounds
tests compiled in (-DCPATTN_CHECKS; see include/cpattn.h). The two compile
in parallel.

Run ``python -m context_blockwise_causal_gb300._build`` or call ``build()``.
"""
import os
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
LIB_PATH = os.path.join(PKG_DIR, "libcpattn.so")
CHECKED_LIB_PATH = os.path.join(PKG_DIR, "libcpattn_checked.so")
SOURCES = ["cpattn_api.cu"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17", "-shared",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]


def _nvcc():
    for cand in (os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"), "nvcc"):
        if os.path.sep not in cand or os.path.exists(cand):
            return cand
    return "nvcc"


def is_stale():
    """True when a library is missing or older than a source or header."""
    if not (os.path.exists(LIB_PATH) and os.path.exists(CHECKED_LIB_PATH)):
        return True
    built = min(os.path.getmtime(LIB_PATH), os.path.getmtime(CHECKED_LIB_PATH))
    inc = os.path.join(os.path.dirname(PKG_DIR), "include")
    for d in (CSRC, inc):
        for f in os.listdir(d):
            if os.path.getmtime(os.path.join(d, f)) > built:
                return True
    return False


def build(verbose=False):
    """Compile every CUDA source of the library into one shared object, and
    the checked build beside it."""
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    jobs = []
    for out, extra in ((LIB_PATH, []), (CHECKED_LIB_PATH, ["-DCPATTN_CHECKS"])):
        cmd = [_nvcc(), *NVCC_FLAGS, *extra, "-o", out + ".tmp", *srcs]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), flush=True)
        jobs.append((out, cmd, subprocess.Popen(cmd)))
    failed = [cmd for _, cmd, proc in jobs if proc.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    for out, _, _ in jobs:
        os.replace(out + ".tmp", out)
    return LIB_PATH


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
    print(LIB_PATH)

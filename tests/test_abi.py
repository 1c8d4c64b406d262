"""CPU tests of the C-ABI library: it loads, exports every function that
include/*.h declares, and its host-only logic behaves (no GPU needed: the
calls below return before touching a device)."""
import ctypes
import glob
import os
import re
import subprocess
import sys

import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import context_blockwise_causal_gb300 as pkg

    from context_blockwise_causal_gb300._build import is_stale

    if is_stale():
        pkg.build()
    return pkg.library()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(cpattn_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("cpattn_fwd", "cpattn_bwd", "cpattn_bwd_workspace_bytes", "cpattn_zigzag_index"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def _declared_arity():
    """Number of parameters of every function the headers declare."""
    out = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for name, params in re.findall(r"\b(cpattn_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
            params = params.strip()
            out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argtypes_match_the_header(lib):
    """Every function the binding declares to ctypes takes as many arguments
    as the header says (a wrong count would shift every later argument)."""
    arity = _declared_arity()
    assert arity, "no declarations parsed"
    for name, n in arity.items():
        fn = getattr(lib, name)
        if fn.argtypes is not None:
            assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)


def test_zigzag_index_matches_oracle(lib):
    from context_blockwise_causal_gb300 import cpattn_zigzag_index

    for s, cp in ((8, 2), (12, 3), (4096, 4), (16384, 8), (96, 3), (2, 1)):
        got = cpattn_zigzag_index(s, cp)
        assert got.shape == (cp, s // cp)
        assert torch.equal(got, oracle.zigzag_global_index(s, cp))  # bit-exact


def test_zigzag_index_errors(lib):
    buf = (ctypes.c_int64 * 64)()
    assert lib.cpattn_zigzag_index(10, 3, buf) == -1  # s not divisible by 2cp
    assert lib.cpattn_zigzag_index(12, 0, buf) == -1
    assert lib.cpattn_zigzag_index(12, 3, None) == -2


def test_selftest_rejects_limits_out_of_range(lib):
    lib.cpattn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    assert lib.cpattn_selftest_wait_timeout(0, None) == -1
    assert lib.cpattn_selftest_wait_timeout(3_000_000_000, None) == -1


def test_strerror_and_version(lib):
    assert lib.cpattn_strerror(0) == b"ok"
    for code in range(-8, 0):
        assert lib.cpattn_strerror(code) not in (b"", b"unknown error")
    assert lib.cpattn_strerror(-99) == b"unknown error"
    assert lib.cpattn_version() >= 100


def test_checked_build_loads_and_reports_itself(lib):
    """The checked build (kernels' bounds tests compiled in) exports the same
    entry points; each build reports which one it is, and the bounds
    self-test refuses to run where no tests were compiled."""
    import context_blockwise_causal_gb300 as pkg

    chk = pkg.checked_library()
    for name in _declared():
        assert hasattr(chk, name), name
    assert lib.cpattn_checked_build() == 0 and chk.cpattn_checked_build() == 1
    assert lib.cpattn_selftest_bounds(None, None, None, None, None, 1, 256, 2, 2, 128, 2, None) == -1


def test_fwd_argument_errors_are_reported_before_any_device_work(lib):
    p = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    f = lib.cpattn_fwd
    assert f(None, p, p, p, p, 1, 512, 4, 4, 64, 2, 1, None) == -2
    assert f(p, p, p, p, p, 1, 512, 4, 4, 96, 2, 1, None) == -1    # unsupported d
    assert f(p, p, p, p, p, 1, 510, 4, 4, 64, 2, 1, None) == -1    # s % 2cp
    assert f(p, p, p, p, p, 1, 512, 6, 4, 64, 2, 1, None) == -1    # hq % hkv
    assert f(p, p, p, p, p, 0, 512, 4, 4, 64, 2, 1, None) == -1
    assert f(p, p, p, p, p, 1, 512, 4, 4, 64, 0, 1, None) == -1
    odd = ctypes.c_void_p(4096 + 8)
    assert f(odd, p, p, p, p, 1, 512, 4, 4, 64, 2, 1, None) == -3  # misaligned


def test_bwd_argument_errors_and_workspace_size(lib):
    n = lib.cpattn_bwd_workspace_bytes(1, 512, 4, 2, 64, 2)
    # two fp32 vectors (L*log2e and D) per query row and head, tile-padded
    assert n == 2 * 4 * 512 * 4
    # ragged chunks pad each chunk to whole 128-row tiles: c = 160 -> 256 rows
    assert lib.cpattn_bwd_workspace_bytes(1, 640, 2, 1, 64, 2) == 2 * 2 * (4 * 256) * 4
    assert lib.cpattn_bwd_workspace_bytes(1, 510, 4, 2, 64, 2) == 0
    p = ctypes.c_void_p(4096)
    b = lib.cpattn_bwd
    assert b(p, p, p, p, p, p, p, p, p, p, n - 1, 1, 512, 4, 2, 64, 2, 1, None) == -5
    assert b(p, p, p, p, p, p, p, p, p, None, n, 1, 512, 4, 2, 64, 2, 1, None) == -2
    assert b(p, p, p, p, p, p, p, p, p, p, n, 1, 512, 4, 3, 64, 2, 1, None) == -1


def test_unfused_argument_errors_and_workspace_size(lib):
    # two fp32 copies of O and of the LSE, each rounded up to 256 bytes
    o_bytes, l_bytes = 1 * 512 * 4 * 64 * 4, 1 * 4 * 512 * 4
    assert lib.cpattn_fwd_unfused_workspace_bytes(1, 512, 4, 64) == 2 * o_bytes + 2 * l_bytes
    assert lib.cpattn_fwd_unfused_workspace_bytes(1, 512, 4, 96) == 0
    n = lib.cpattn_fwd_unfused_workspace_bytes(1, 512, 4, 64)
    p = ctypes.c_void_p(4096)
    u = lib.cpattn_fwd_unfused
    assert u(p, p, p, p, p, p, n - 1, 1, 512, 4, 4, 64, 2, 1, None) == -5
    assert u(p, p, p, p, p, None, n, 1, 512, 4, 4, 64, 2, 1, None) == -2
    assert u(p, p, p, p, p, ctypes.c_void_p(4096 + 16), n, 1, 512, 4, 4, 64, 2, 1, None) == -3
    assert u(p, p, p, p, p, p, n, 1, 512, 4, 3, 64, 2, 1, None) == -1
    st = lib.cpattn_fwd_step
    assert st(p, p, p, p, p, 1, 512, 4, 4, 64, 2, 2, 1, None) == -1   # step >= cp
    assert st(p, p, p, p, p, 1, 512, 4, 4, 64, 2, -1, 1, None) == -1
    assert st(p, p, p, None, p, 1, 512, 4, 4, 64, 2, 0, 1, None) == -2
    m = lib.cpattn_lse_merge
    assert m(p, p, p, None, p, p, None, 1, 512, 4, 64, None) == -2   # o_b without lse_b
    assert m(p, p, None, None, None, p, None, 1, 512, 4, 64, None) == -2  # no output
    assert m(p, p, None, None, p, p, None, 1, 512, 4, 96, None) == -1
    assert m(ctypes.c_void_p(4096 + 4), p, None, None, p, p, None, 1, 512, 4, 64, None) == -3


def test_rope_argument_errors(lib):
    p = ctypes.c_void_p(4096)
    r = lib.cpattn_rope
    assert r(None, 1, 512, 4, 64, 512, 2, -1, None, 0, 10000.0, 0, None) == -2
    assert r(p, 1, 512, 4, 96, 512, 2, -1, None, 0, 10000.0, 0, None) == -1   # d
    assert r(p, 1, 500, 4, 64, 512, 2, -1, None, 0, 10000.0, 0, None) == -1   # natural order: n == s
    assert r(p, 1, 512, 4, 64, 512, 2, 0, None, 0, 10000.0, 0, None) == -1    # shard: n == s / cp
    assert r(p, 1, 256, 4, 64, 512, 2, 2, None, 0, 10000.0, 0, None) == -1    # rank >= cp
    assert r(p, 2, 512, 4, 64, 512, 2, -1, p, 3, 10000.0, 0, None) == -1      # packing needs b == 1
    assert r(p, 1, 512, 4, 64, 512, 2, -1, None, 0, 1.0, 0, None) == -1      # base > 1
    assert r(ctypes.c_void_p(4096 + 4), 1, 512, 4, 64, 512, 2, -1, None, 0, 10000.0, 0, None) == -3


def test_scaled_entry_points_reject_bad_scales(lib):
    p = ctypes.c_void_p(4096)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert lib.cpattn_fwd_ex(p, p, p, p, p, 1, 512, 4, 4, 64, 2, 1, bad, None) == -1
        assert lib.cpattn_bwd_ex(p, p, p, p, p, p, p, p, p, p, 1 << 20, 1, 512, 4, 2, 64, 2, 1, bad, None) == -1


def test_varlen_offsets_are_checked(lib):
    p = ctypes.c_void_p(4096)
    f = lib.cpattn_fwd_varlen

    def cu(*xs):
        return (ctypes.c_int * len(xs))(*xs)

    assert f(p, p, p, p, p, None, 1, 4, 4, 64, 2, 1, 0.0, None) == -2
    assert f(p, p, p, p, p, cu(0, 510), 1, 4, 4, 64, 2, 1, 0.0, None) == -1      # 510 % 4
    assert f(p, p, p, p, p, cu(4, 512), 1, 4, 4, 64, 2, 1, 0.0, None) == -1      # cu[0] != 0
    assert f(p, p, p, p, p, cu(0, 512, 256), 2, 4, 4, 64, 2, 1, 0.0, None) == -1  # decreasing
    assert f(p, p, p, p, p, cu(0, 512), 1, 4, 4, 64, 2, 1, -1.0, None) == -1     # scale
    w = lib.cpattn_bwd_varlen_workspace_bytes
    # one launch for all samples: two fp32 vectors per (sample, head), each
    # sample's rows padded to the longest sample's tiles (here 2 per chunk:
    # 2cp * 2 * 128 = 1024 rows)
    assert w(cu(0, 512, 1536, 1792), 3, 4, 2, 64, 2) == 2 * 3 * 4 * 1024 * 4
    assert w(cu(0, 510), 1, 4, 2, 64, 2) == 0


def test_sizes_beyond_the_index_range_are_rejected(lib):
    p = ctypes.c_void_p(4096)
    # b * s >= 2^31 tokens: 32-bit token indices would overflow
    assert lib.cpattn_fwd(p, p, p, p, p, 2, 1 << 30, 1, 1, 64, 1, 1, None) == -1
    assert lib.cpattn_bwd_workspace_bytes(2, 1 << 30, 1, 1, 64, 1) == 0
    assert lib.cpattn_fwd_unfused(p, p, p, p, p, p, 1 << 40, 2, 1 << 30, 1, 1, 64, 1, 1, None) == -1
    # a sequence just below 2^31 tokens whose tile padding would not fit an int
    s = (1 << 31) - 2
    assert lib.cpattn_fwd(p, p, p, p, p, 1, s, 1, 1, 64, 1, 1, None) == -1
    assert lib.cpattn_bwd_workspace_bytes(1, s, 1, 1, 64, 1) == 0


def test_product_fails_loudly_without_the_library(tmp_path):
    """With the library absent, the binding's entry points raise: no CPU or
    PyTorch fallback answers in its place. Run in a fresh interpreter whose
    package points at a path with no library."""
    code = f"""
import context_blockwise_causal_gb300 as pkg
import torch
pkg.LIB_PATH = {str(tmp_path / 'libcpattn.so')!r}
pkg._LIB = None
q = torch.zeros(1, 256, 2, 64, dtype=torch.bfloat16)
calls = {{
    "library": lambda: pkg.library(),
    "cpattn_zigzag_index": lambda: pkg.cpattn_zigzag_index(256, 2),
    "cpattn_fwd": lambda: pkg.cpattn_fwd(q, q, q, 2),
}}
for name, call in calls.items():
    try:
        call()
    except (RuntimeError, TypeError, ValueError) as e:
        print(name, type(e).__name__, "missing" in str(e) or "CUDA" in str(e))
    else:
        print(name, "returned")
"""
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = dict(ln.split(" ", 1) for ln in r.stdout.strip().splitlines())
    assert lines["library"] == "RuntimeError True"
    assert lines["cpattn_zigzag_index"] == "RuntimeError True"
    # a CPU tensor is refused before the library is reached; either way nothing computes it
    assert not lines["cpattn_fwd"].startswith("returned")


def test_grid_cap_argument(lib):
    assert lib.cpattn_set_max_ctas(-1) == -1  # CPATTN_ERR_INVALID_ARG
    assert lib.cpattn_set_max_ctas(37) == 0
    assert lib.cpattn_set_max_ctas(0) == 0

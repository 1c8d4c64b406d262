"""The C ABI used from plain C: tests/c_abi_client.c is compiled with gcc as
C99 against include/cpattn.h and the CUDA runtime header, warnings as errors,
and linked with libcpattn.so.

On the CPU the client runs its host-only calls (version, zigzag index map,
argument errors, workspace size). On the GPU it runs the forward and backward
on device buffers of its own; its outputs are compared with the CPU fp64
oracle (the same bars as the Python-side parity tests: O within 1e-2 beyond
bf16 output rounding, LSE within 1e-3, gradients within 2e-2 relative L2) and,
bit for bit, with the same calls made through the Python binding.
"""
import os
import subprocess

import pytest
import torch

import oracle
from context_blockwise_causal_gb300.workloads import Workload, make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    import context_blockwise_causal_gb300 as pkg
    from context_blockwise_causal_gb300._build import LIB_PATH, is_stale

    if is_stale():
        pkg.build()
    pkg_dir = os.path.dirname(LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_client") / "c_abi_client")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O1",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(CUDA_HOME, "include"),
           os.path.join(ROOT, "tests", "c_abi_client.c"), "-o", exe,
           "-L", pkg_dir, "-lcpattn", f"-Wl,-rpath,{pkg_dir}",
           "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA_HOME, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_client_host_calls(client):
    out = subprocess.run([client], check=True, capture_output=True, text=True, timeout=60).stdout
    lines = dict(line.split(" ", 1) for line in out.strip().splitlines())
    zz = [int(t) for t in lines["zigzag"].split()]
    assert zz == oracle.zigzag_global_index(8, 2).reshape(-1).tolist()
    assert lines["null"].startswith("pointers -> -2 ")
    assert lines["s"].startswith("not divisible by 2cp -> -1 ")
    assert int(lines["bwd"].rsplit(":", 1)[1].split()[0]) > 0


def _raw(t):
    return t.contiguous().view(torch.uint8).numpy().tobytes()


def _load(path, dtype, shape):
    data = bytearray(open(path, "rb").read())
    return torch.frombuffer(data, dtype=dtype).reshape(shape).clone()


@pytest.mark.gpu
def test_c_client_fwd_bwd_matches_oracle_and_binding(client, tmp_path):
    from context_blockwise_causal_gb300 import cpattn_bwd, cpattn_fwd

    # GQA (3 query heads per KV head), batch 2, ragged tiles (c = 160), cp 3
    w = Workload("c_client", b=2, s=960, hq=6, hkv=2, d=128, cp=3, causal=True, backward=True, seed=29)
    x = make_inputs(w, device="cpu")
    for name in ("q", "k", "v", "do"):
        (tmp_path / f"{name}.bin").write_bytes(_raw(x[name]))
    run = subprocess.run([client, "gpu", str(tmp_path), str(w.b), str(w.s), str(w.hq), str(w.hkv), str(w.d),
                          str(w.cp)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "gpu run ok" in run.stdout
    qs, ks = (w.b, w.s, w.hq, w.d), (w.b, w.s, w.hkv, w.d)
    o = _load(tmp_path / "o.bin", torch.bfloat16, qs)
    lse = _load(tmp_path / "lse.bin", torch.float32, (w.b, w.hq, w.s))
    dq = _load(tmp_path / "dq.bin", torch.bfloat16, qs)
    dk = _load(tmp_path / "dk.bin", torch.bfloat16, ks)
    dv = _load(tmp_path / "dv.bin", torch.bfloat16, ks)

    o_ref, l_ref = oracle.attention_forward(x["q"], x["k"], x["v"], causal=True)
    err = (o.double() - o_ref).abs() - o_ref.abs() * 2.0**-9
    assert err.max().item() <= 1e-2
    assert (lse.double() - l_ref).abs().max().item() <= 1e-3
    refs = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], causal=True)
    for name, got, ref in (("dq", dq, refs[0]), ("dk", dk, refs[1]), ("dv", dv, refs[2])):
        rel = ((got.double() - ref).norm() / ref.norm()).item()
        assert rel <= 2e-2, f"{name} rel L2 {rel:.3e}"

    g = {n: t.cuda() for n, t in x.items()}
    o_b, l_b = cpattn_fwd(g["q"], g["k"], g["v"], w.cp, causal=True)
    dq_b, dk_b, dv_b = cpattn_bwd(g["q"], g["k"], g["v"], o_b, l_b, g["do"], w.cp, causal=True)
    torch.cuda.synchronize()
    for got, ref in ((o, o_b), (lse, l_b), (dq, dq_b), (dk, dk_b), (dv, dv_b)):
        assert torch.equal(got, ref.cpu())

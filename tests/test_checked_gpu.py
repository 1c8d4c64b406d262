"""The checked build on the GPU: libcpattn_checked.so, whose kernels test
every global access against the extents of the buffers (bit 20 of the
device status word; stores out of range skipped, bulk copies kept inside).

On valid calls no test may fire and every output must equal the normal
build's bit for bit: the tests add no arithmetic. The bounds self-test then
makes them fire on purpose (the forward told that q and o hold one row fewer
than they do; the buffers hold it, so nothing is touched outside them).
"""
import ctypes

import pytest
import torch

import context_blockwise_causal_gb300 as pkg
from context_blockwise_causal_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

BOUNDS_BIT = 1 << 20


def _status(lib):
    st = ctypes.c_int(0)
    lib.cpattn_device_status(None, ctypes.byref(st))
    return st.value


def _fwd_bwd(lib, x, w):
    b, s, hq, hkv, d, cp = w.b, w.s, w.hq, w.hkv, w.d, w.cp
    o = torch.full_like(x["q"], 7.0)
    lse = torch.full((b, hq, s), 7.0, device="cuda")
    dq, dk, dv = (torch.full_like(x[n], 7.0) for n in ("q", "k", "v"))
    n = pkg.cpattn_bwd_workspace_bytes(b, s, hq, hkv, d, cp)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    assert lib.cpattn_fwd(p(x["q"]), p(x["k"]), p(x["v"]), p(o), p(lse), b, s, hq, hkv, d, cp, int(w.causal),
                          None) == 0
    assert lib.cpattn_bwd(p(x["q"]), p(x["k"]), p(x["v"]), p(o), p(lse), p(x["do"]), p(dq), p(dk), p(dv), p(ws), n,
                          b, s, hq, hkv, d, cp, int(w.causal), None) == 0
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


GEOMS = [
    # b, s, hq, hkv, d, cp, causal
    (1, 960, 6, 2, 128, 3, True),     # ragged tiles (c = 160), G = 3
    (2, 1024, 4, 2, 128, 2, True),    # GQA head pairs
    (1, 2048, 4, 4, 128, 4, True),    # MHA: tile pairs
    (1, 768, 4, 4, 128, 3, False),    # no mask
    (1, 1536, 4, 4, 64, 3, True),     # d = 64
    (3, 8, 2, 1, 128, 4, True),       # one token per half-chunk
]


@pytest.mark.parametrize("b,s,hq,hkv,d,cp,causal", GEOMS)
def test_checked_build_is_silent_and_bit_identical(b, s, hq, hkv, d, cp, causal):
    w = Workload("chk", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, causal=causal, backward=True, seed=3 + s)
    x = make_inputs(w, device="cuda")
    lib, chk = pkg.library(), pkg.checked_library()
    ref = _fwd_bwd(lib, x, w)
    assert _status(lib) == 0
    got = _fwd_bwd(chk, x, w)
    assert _status(chk) == 0, hex(_status(chk))
    for name, r, g in zip(("o", "lse", "dq", "dk", "dv"), ref, got):
        assert torch.equal(r, g), name


def test_checked_build_packed_samples_and_rank_local():
    """Packed samples (sample offsets, per-sample tiles) and one rank's share
    of a CP group (local query rows, rank-major K/V shards): no test fires."""
    chk = pkg.checked_library()
    hq, hkv, d, cp = 4, 2, 128, 2
    lens = [256, 0, 640, 384]
    cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0)), dtype=torch.int32)
    total = int(cu[-1])
    gen = torch.Generator(device="cuda").manual_seed(11)
    q = torch.randn(total, hq, d, generator=gen, device="cuda").bfloat16()
    k = torch.randn(total, hkv, d, generator=gen, device="cuda").bfloat16()
    v = torch.randn(total, hkv, d, generator=gen, device="cuda").bfloat16()
    do = torch.randn(total, hq, d, generator=gen, device="cuda").bfloat16()
    o, lse = torch.empty_like(q), torch.empty(hq, total, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    cu_h = (ctypes.c_int * len(cu))(*cu.tolist())
    n = chk.cpattn_bwd_varlen_workspace_bytes(cu_h, len(lens), hq, hkv, d, cp)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    scale = ctypes.c_float(d ** -0.5)
    assert chk.cpattn_fwd_varlen(p(q), p(k), p(v), p(o), p(lse), cu_h, len(lens), hq, hkv, d, cp, 1, scale, None) == 0
    assert chk.cpattn_bwd_varlen(p(q), p(k), p(v), p(o), p(lse), p(do), p(dq), p(dk), p(dv), p(ws), n, cu_h,
                                 len(lens), hq, hkv, d, cp, 1, scale, None) == 0
    torch.cuda.synchronize()
    assert _status(chk) == 0, hex(_status(chk))
    # rank 1 of a 2-rank group, the K/V shards gathered rank-major
    w = Workload("rk", b=1, s=1024, hq=4, hkv=2, d=128, cp=2, backward=True, seed=5)
    x = make_inputs(w, device="cuda")
    from context_blockwise_causal_gb300.cp_group import zigzag_shard
    sh = {nm: [zigzag_shard(x[nm], w.cp, r) for r in range(w.cp)] for nm in ("q", "k", "v", "do")}
    k_all, v_all = torch.stack(sh["k"]).contiguous(), torch.stack(sh["v"]).contiguous()
    q1, do1 = sh["q"][1].contiguous(), sh["do"][1].contiguous()
    o1, l1 = torch.empty_like(q1), torch.empty(1, w.hq, q1.shape[1], device="cuda")
    assert chk.cpattn_fwd_rank(p(q1), p(k_all), p(v_all), p(o1), p(l1), 1, w.s, w.hq, w.hkv, w.d, w.cp, 1, 1,
                               scale, None) == 0
    nw = chk.cpattn_bwd_rank_workspace_bytes(1, w.s, w.hq, w.hkv, w.d, w.cp)
    wsr = torch.empty(nw, dtype=torch.uint8, device="cuda")
    dq1, dkp, dvp = torch.empty_like(q1), torch.empty_like(k_all), torch.empty_like(v_all)
    assert chk.cpattn_bwd_rank(p(q1), p(k_all), p(v_all), p(o1), p(l1), p(do1), p(dq1), p(dkp), p(dvp), p(wsr), nw,
                               1, w.s, w.hq, w.hkv, w.d, w.cp, 1, 1, scale, None) == 0
    torch.cuda.synchronize()
    assert _status(chk) == 0, hex(_status(chk))


def test_bounds_self_test_fires_and_clears():
    chk = pkg.checked_library()
    w = Workload("bnd", b=1, s=512, hq=4, hkv=2, d=128, cp=2, seed=9)
    x = make_inputs(w, device="cuda", with_grad=False)
    o = torch.zeros_like(x["q"])
    lse = torch.zeros(w.b, w.hq, w.s, device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    assert chk.cpattn_selftest_bounds(p(x["q"]), p(x["k"]), p(x["v"]), p(o), p(lse), w.b, w.s, w.hq, w.hkv, w.d,
                                      w.cp, None) == 0
    torch.cuda.synchronize()
    st = ctypes.c_int(0)
    assert chk.cpattn_device_status(None, ctypes.byref(st)) == -7  # the status word was non-zero
    assert st.value & BOUNDS_BIT, hex(st.value)
    assert not o[0, -1].any()  # the last row's stores were skipped
    assert _status(chk) == 0  # read and cleared

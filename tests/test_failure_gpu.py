"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up, the kernel records it in the device status word and
returns, and the context stays usable for real work."""
import ctypes

import pytest
import torch

import oracle
from context_blockwise_causal_gb300 import cpattn_device_status, cpattn_fwd, cpattn_selftest_wait_timeout
from context_blockwise_causal_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_survives():
    assert cpattn_device_status() == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    cpattn_selftest_wait_timeout(20_000_000)  # 20 ms
    e1.record()
    e1.synchronize()
    assert e0.elapsed_time(e1) >= 19.0  # it did wait out its limit
    status = cpattn_device_status()
    assert status & 0x10000, hex(status)
    assert cpattn_device_status() == 0  # read and cleared
    # a real launch afterwards runs and is correct
    w = Workload("after", b=1, s=512, hq=4, hkv=2, d=128, cp=2, seed=3)
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], w.cp)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    o_ref, l_ref = oracle.attention_forward(x["q"].cpu(), x["k"].cpu(), x["v"].cpu())
    assert (lse.double().cpu() - l_ref).abs().max().item() <= 1e-3
    assert (o.double().cpu() - o_ref).abs().max().item() <= 2e-2


def test_kernels_abort_mid_run_and_drain_their_own_work():
    """The attention kernels' own abort path: with the producers' waits for free
    buffers limited to 1 ns, a producer in every CTA gives up mid-run. The
    status word must show the producers' bits (forward 0, backward 8) and not
    the drain bits (3, 12): every role waited for its own copies and MMAs
    before the CTA released memory. A normal forward and backward afterwards
    still match the oracle, so the context is intact."""
    from context_blockwise_causal_gb300 import cpattn_bwd, cpattn_bwd_workspace_bytes, library

    lib = library()
    w = Workload("abort", b=1, s=4096, hq=8, hkv=2, d=128, cp=2, backward=True, seed=77)
    x = make_inputs(w, device="cuda")
    o = torch.empty_like(x["q"])
    lse = torch.empty(1, 8, 4096, device="cuda")
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    n = cpattn_bwd_workspace_bytes(1, 4096, 8, 2, 128, 2)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    assert cpattn_device_status() == 0
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.cpattn_selftest_abort(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), x["do"].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                   ws.data_ptr(), n, 1, 4096, 8, 2, 128, 2, 1, st)
    assert rc == 0, lib.cpattn_strerror(rc)
    torch.cuda.synchronize()
    status = cpattn_device_status()
    assert status & (1 << 0) and status & (1 << 8), hex(status)
    assert not status & ((1 << 3) | (1 << 12) | (1 << 11)), hex(status)
    # the context still works: a normal forward and backward against the oracle
    small = Workload("after", b=1, s=1024, hq=4, hkv=2, d=128, cp=2, backward=True, seed=78)
    y = make_inputs(small, device="cuda")
    o2, l2 = cpattn_fwd(y["q"], y["k"], y["v"], 2)
    g = cpattn_bwd(y["q"], y["k"], y["v"], o2, l2, y["do"], 2)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    cpu = {k_: t.cpu() for k_, t in y.items()}
    o_ref, l_ref = oracle.attention_forward(cpu["q"], cpu["k"], cpu["v"])
    assert (l2.cpu().double() - l_ref).abs().max().item() <= 1e-3
    grads = oracle.attention_backward(cpu["q"], cpu["k"], cpu["v"], cpu["do"])
    for got, ref in zip(g, grads):
        assert ((got.double().cpu() - ref).norm() / ref.norm()).item() <= 2e-2


def test_abort_selftest_rejects_a_bad_limit():
    from context_blockwise_causal_gb300 import library

    lib = library()
    p = ctypes.c_void_p(4096)  # never dereferenced: the checks come first
    for limit in (0, 2_000_000_000, 3_000_000_000):  # outside 1 .. 2e9 - 1
        assert lib.cpattn_selftest_abort(p, p, p, p, p, p, p, p, p, p, 1 << 20, 1, 256, 4, 2, 128, 1, limit, None) == -1
    # shapes the self-test kernels are not built for: d = 64, odd head groups
    assert lib.cpattn_selftest_abort(p, p, p, p, p, p, p, p, p, p, 1 << 20, 1, 256, 4, 2, 64, 1, 1000, None) == -1
    assert lib.cpattn_selftest_abort(p, p, p, p, p, p, p, p, p, p, 1 << 20, 1, 256, 3, 1, 128, 1, 1000, None) == -1

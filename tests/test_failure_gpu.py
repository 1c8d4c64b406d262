"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up, the kernel records it in the device status word and
returns, and the context stays usable for real work."""
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

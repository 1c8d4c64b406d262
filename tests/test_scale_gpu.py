"""A caller-chosen softmax scale (cpattn_fwd_ex / cpattn_bwd_ex) through the
C ABI against the CPU fp64 oracle with the same scale. Tolerances as the
default-scale tests: max |O err| <= 1e-2 beyond the bf16 output's half ulp,
max |LSE err| <= 1e-3, relative L2 <= 2e-2 per gradient."""
import pytest
import torch

import oracle
from context_blockwise_causal_gb300 import cpattn_bwd, cpattn_device_status, cpattn_fwd
from context_blockwise_causal_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _half_ulp_bf16(x):
    e = torch.floor(torch.log2(x.abs().clamp_min(2.0 ** -126)))
    return 2.0 ** (e - 8)


def _rel(x, ref):
    x = x.double()
    return ((x - ref).norm() / ref.norm().clamp_min(1e-30)).item()


@pytest.mark.parametrize("b,s,hq,hkv,d,cp,scale", [(1, 512, 4, 2, 128, 2, 0.05), (1, 960, 6, 2, 64, 3, 0.3),
                                                   (2, 768, 4, 4, 128, 3, 1.0 / 128)])
def test_custom_scale_forward_and_backward(b, s, hq, hkv, d, cp, scale):
    w = Workload("scale", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, backward=True, seed=31 + s)
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], cp, scale=scale)
    dq, dk, dv = cpattn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], cp, scale=scale)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    cpu = {k: t.cpu() for k, t in x.items()}
    o_r, l_r = oracle.attention_forward(cpu["q"], cpu["k"], cpu["v"], scale=scale)
    err = (o.double().cpu() - o_r).abs()
    assert (err <= 1e-2 + _half_ulp_bf16(o_r)).all(), err.max().item()
    assert (lse.double().cpu() - l_r).abs().max().item() <= 1e-3
    dq_r, dk_r, dv_r = oracle.attention_backward(cpu["q"], cpu["k"], cpu["v"], cpu["do"], scale=scale)
    for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        assert _rel(got.float().cpu(), ref) <= 2e-2, name


def test_default_scale_through_ex_agrees():
    # 1/sqrt(d) passed as a float differs from the built-in default only in
    # the last bit of the scale
    w = Workload("scale_default", b=1, s=512, hq=4, hkv=2, d=128, cp=2, backward=True, seed=77)
    x = make_inputs(w, device="cuda")
    sc = 1.0 / 128 ** 0.5
    o1, l1 = cpattn_fwd(x["q"], x["k"], x["v"], 2)
    o2, l2 = cpattn_fwd(x["q"], x["k"], x["v"], 2, scale=sc)
    g1 = cpattn_bwd(x["q"], x["k"], x["v"], o1, l1, x["do"], 2)
    g2 = cpattn_bwd(x["q"], x["k"], x["v"], o1, l1, x["do"], 2, scale=sc)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2 * _half_ulp_bf16(o1.double()).max().item()
    assert (l1 - l2).abs().max().item() <= 1e-5
    for a, b in zip(g1, g2):
        assert _rel(a.float(), b.double()) <= 1e-2

"""The unfused forward (one launch per CP step + log-sum-exp merges), through
the C ABI, against the CPU fp64 oracle.

* cpattn_fwd_step: every step's partial O (fp32, max |err| <= 1e-2) and LSE
  (<= 1e-3) against the oracle's per-step partials (oracle.cp_step_partials),
  including the rows that take no part in the step (O = 0, L = -inf).
* cpattn_lse_merge: random partials against oracle.lse_merge, in place.
* cpattn_fwd_unfused: the merged result against uncut attention, with the
  fused forward's tolerances (max |O err| <= 1e-2 beyond the bf16 output's
  own half-ulp rounding; max |LSE err| <= 1e-3).
"""
import math

import pytest
import torch

import oracle
from context_blockwise_causal_gb300 import (cpattn_device_status, cpattn_fwd, cpattn_fwd_step, cpattn_fwd_unfused,
                                            cpattn_lse_merge)
from context_blockwise_causal_gb300.workloads import WORKLOADS, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL = 1e-2, 1e-3
# A step's partial O is an attention output over the block's keys, formed
# the same way as the fused forward's (P rounded to bf16 for P.V, fp32
# accumulation), only stored in fp32: the same 1e-2 bound, with no output
# rounding to add.
PART_TOL = O_TOL


def _half_ulp_bf16(x):
    e = torch.floor(torch.log2(x.abs().clamp_min(2.0 ** -126)))
    return 2.0 ** (e - 8)


SMALL = [
    # b, s, hq, hkv, d, cp, causal
    (1, 512, 4, 4, 64, 2, True),
    (2, 1024, 4, 2, 128, 4, True),
    (1, 960, 6, 2, 128, 3, True),    # ragged tiles (c = 160), G = 3
    (1, 640, 3, 1, 64, 2, True),     # odd hq, MQA, ragged
    (1, 768, 4, 4, 128, 3, False),   # no mask
    (1, 256, 2, 2, 128, 1, True),    # cp = 1
    (1, 2048, 2, 2, 128, 2, True),   # MHA, two tiles per chunk: tile-pair units in every step
    (1, 1536, 3, 1, 64, 3, False),   # G = 3, c = 256: tile pairs without the mask
]


@pytest.mark.parametrize("b,s,hq,hkv,d,cp,causal", SMALL)
def test_step_partials_match_oracle(b, s, hq, hkv, d, cp, causal):
    w = Workload("step", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, causal=causal, seed=5 + s + cp)
    x = make_inputs(w, device="cuda")
    cpu = {k: t.cpu().double() for k, t in x.items()}
    for i in range(cp):
        o_i, l_i = cpattn_fwd_step(x["q"], x["k"], x["v"], cp, i, causal=causal)
        torch.cuda.synchronize()
        assert cpattn_device_status() == 0
        o_r, l_r = oracle.cp_step_partials(cpu["q"], cpu["k"], cpu["v"], cp, i, causal=causal)
        l_i = l_i.double().cpu()
        o_i = o_i.double().cpu()
        absent = torch.isinf(l_r)
        assert torch.equal(torch.isinf(l_i), absent), f"step {i}: rows taking part differ"
        assert (l_i[absent] < 0).all()
        assert (o_i.permute(0, 2, 1, 3)[absent] == 0).all()
        assert (l_i[~absent] - l_r[~absent]).abs().max().item() <= LSE_TOL, f"step {i} lse"
        assert (o_i - o_r).abs().max().item() <= PART_TOL, f"step {i} o"


def test_lse_merge_matches_oracle_in_place():
    g = torch.Generator(device="cpu").manual_seed(17)
    b, s, hq, d = 2, 384, 3, 128
    o_a = torch.randn(b, s, hq, d, generator=g)
    o_b = torch.randn(b, s, hq, d, generator=g)
    l_a = torch.randn(b, hq, s, generator=g) * 4
    l_b = torch.randn(b, hq, s, generator=g) * 4
    l_a[0, 0, :7] = -math.inf        # rows one side has not seen
    l_b[1, 2, 5:9] = -math.inf
    l_a[1, 1, 3] = l_b[1, 1, 3] = -math.inf   # neither side
    o_a[0, :7, 0] = 0
    o_b[1, 5:9, 2] = 0
    o_a[1, 3, 1] = o_b[1, 3, 1] = 0
    dev = {k: t.cuda() for k, t in dict(o_a=o_a, o_b=o_b, l_a=l_a, l_b=l_b).items()}
    o_out, l_out, o16 = cpattn_lse_merge(dev["o_a"], dev["l_a"], dev["o_b"], dev["l_b"], o_out=dev["o_a"],
                                         lse_out=dev["l_a"], o_bf16=torch.empty(b, s, hq, d, device="cuda",
                                                                                dtype=torch.bfloat16))
    torch.cuda.synchronize()
    for bi in range(b):
        for h in range(hq):
            O, L = oracle.lse_merge([(o_a[bi, :, h].double(), l_a[bi, h].double()),
                                     (o_b[bi, :, h].double(), l_b[bi, h].double())])
            got_l = l_out[bi, h].double().cpu()
            fin = torch.isfinite(L)
            assert torch.equal(torch.isfinite(got_l), fin)
            assert (got_l[fin] - L[fin]).abs().max().item() <= 1e-5
            got_o = o_out[bi, :, h].double().cpu()
            assert (got_o - O).abs().max().item() <= 1e-5
            assert (o16[bi, :, h].double().cpu() - O).abs().max().item() <= 1e-5 + _half_ulp_bf16(O).max().item()


@pytest.mark.parametrize("b,s,hq,hkv,d,cp,causal", SMALL)
def test_unfused_forward_matches_oracle(b, s, hq, hkv, d, cp, causal):
    w = Workload("unfused", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, causal=causal, seed=9 + s + cp)
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd_unfused(x["q"], x["k"], x["v"], cp, causal=causal)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    o_r, l_r = oracle.attention_forward(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), causal=causal)
    err = (o.double().cpu() - o_r).abs()
    assert (err <= O_TOL + _half_ulp_bf16(o_r)).all(), err.max().item()
    assert (lse.double().cpu() - l_r).abs().max().item() <= LSE_TOL
    # and it agrees with the fused forward
    o_f, l_f = cpattn_fwd(x["q"], x["k"], x["v"], cp, causal=causal)
    torch.cuda.synchronize()
    assert (o_f.float() - o.float()).abs().max().item() <= 2 * O_TOL
    assert (l_f - lse).abs().max().item() <= LSE_TOL


def test_unfused_forward_full_size_gqa():
    w = WORKLOADS["gqa_b1_s16384_h64kv8_d128_cp8"]
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd_unfused(x["q"], x["k"], x["v"], w.cp, causal=w.causal)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    rows = sample_rows(w, w.check_rows, seed=w.seed + 5)
    cpu = {k: t.cpu() for k, t in x.items()}
    o_r, l_r = oracle.attention_forward(cpu["q"], cpu["k"], cpu["v"], causal=w.causal, rows=rows)
    err = (o.double().cpu()[:, rows] - o_r).abs()
    assert (err <= O_TOL + _half_ulp_bf16(o_r)).all(), err.max().item()
    assert (lse.double().cpu()[:, :, rows] - l_r).abs().max().item() <= LSE_TOL

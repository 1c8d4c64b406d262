"""Packed samples (cpattn_fwd_varlen / cpattn_bwd_varlen) through the C ABI
against the CPU fp64 oracle (oracle.varlen_attention_*): mixed lengths,
empty samples, ragged tiles, GQA, d = 64 and 128, a custom scale, with and
without the causal mask.
Tolerances as for one sequence: max |O err| <= 1e-2 beyond the bf16
output's half ulp, max |LSE err| <= 1e-3, relative L2 <= 2e-2 per gradient."""
import pytest
import torch

import oracle
from context_blockwise_causal_gb300 import cpattn_bwd_varlen, cpattn_device_status, cpattn_fwd_varlen

pytestmark = pytest.mark.gpu


def _half_ulp_bf16(x):
    e = torch.floor(torch.log2(x.abs().clamp_min(2.0 ** -126)))
    return 2.0 ** (e - 8)


def _rel(x, ref):
    x = x.double()
    return ((x - ref).norm() / ref.norm().clamp_min(1e-30)).item()


CASES = [
    # lengths, hq, hkv, d, cp, scale, causal
    ([512, 1024, 256], 4, 2, 128, 2, None, True),
    ([960, 0, 192, 384], 6, 2, 64, 3, None, True),     # empty sample, ragged chunks
    ([2048, 128], 8, 1, 128, 4, 0.05, True),          # MQA, custom scale
    ([96], 2, 2, 128, 3, None, True),                 # one sample, c = 16
    ([4, 8, 0, 4], 2, 1, 128, 2, None, True),         # one- and two-token chunks
    ([640, 0, 384, 1152], 4, 2, 128, 2, None, False),  # no mask: every key of the sample
    ([96, 32, 480], 3, 1, 64, 4, 0.1, False),          # no mask, ragged chunks, custom scale
]


@pytest.mark.parametrize("lengths,hq,hkv,d,cp,scale,causal", CASES)
def test_varlen_forward_backward(lengths, hq, hkv, d, cp, scale, causal):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    total = cu[-1]
    g = torch.Generator(device="cpu").manual_seed(100 + total + cp)
    q = torch.randn(total, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(total, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(total, hkv, d, generator=g).to(torch.bfloat16)
    do = torch.randn(total, hq, d, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = cpattn_fwd_varlen(qd, kd, vd, cu, cp, causal=causal, scale=scale)
    dq, dk, dv = cpattn_bwd_varlen(qd, kd, vd, o, lse, dod, cu, cp, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    o_r, l_r = oracle.varlen_attention_forward(q, k, v, cu, causal=causal, scale=scale)
    err = (o.double().cpu() - o_r).abs()
    assert (err <= 1e-2 + _half_ulp_bf16(o_r)).all(), err.max().item()
    assert (lse.double().cpu() - l_r).abs().max().item() <= 1e-3
    dq_r, dk_r, dv_r = oracle.varlen_attention_backward(q, k, v, do, cu, causal=causal, scale=scale)
    for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        assert _rel(got.float().cpu(), ref) <= 2e-2, name


def test_many_short_samples_in_one_launch():
    # 40 samples of 64..1024 tokens (cp = 2): one launch per kernel
    g = torch.Generator(device="cpu").manual_seed(5)
    lens = [int(x) * 64 for x in torch.randint(1, 17, (40,), generator=g)]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    total, hq, hkv, d, cp = cu[-1], 4, 2, 128, 2
    q = torch.randn(total, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(total, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(total, hkv, d, generator=g).to(torch.bfloat16)
    do = torch.randn(total, hq, d, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = cpattn_fwd_varlen(qd, kd, vd, cu, cp)
    dq, dk, dv = cpattn_bwd_varlen(qd, kd, vd, o, lse, dod, cu, cp)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    o_r, l_r = oracle.varlen_attention_forward(q, k, v, cu)
    err = (o.double().cpu() - o_r).abs()
    assert (err <= 1e-2 + _half_ulp_bf16(o_r)).all(), err.max().item()
    assert (lse.double().cpu() - l_r).abs().max().item() <= 1e-3
    dq_r, dk_r, dv_r = oracle.varlen_attention_backward(q, k, v, do, cu)
    for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        assert _rel(got.float().cpu(), ref) <= 2e-2, name


def _packed_case(lens, hq, hkv, d, seed):
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    total = cu[-1]
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(total, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(total, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(total, hkv, d, generator=g).to(torch.bfloat16)
    do = torch.randn(total, hq, d, generator=g).to(torch.bfloat16)
    return cu, q, k, v, do


@pytest.mark.parametrize("cp,hq,hkv,d", [(1, 4, 2, 64), (2, 2, 1, 128)])
def test_more_samples_than_one_launch_holds(cp, hq, hkv, d):
    """More than 512 samples: the library runs consecutive groups of up to
    512, one launch per group, each addressing its rows, its LSE columns
    (lse + the group's first token, row stride the packed total), its sample
    offsets relative to that token and the shared workspace itself. 600
    samples of 0..64 tokens; with cp = 1 the lengths are even but not all
    multiples of 4, so the second group starts at an LSE column that need not
    be 16-byte aligned. Every element against the oracle."""
    g = torch.Generator(device="cpu").manual_seed(600 + cp)
    unit = 2 * cp
    lens = [int(x) * unit for x in torch.randint(0, 64 // unit + 1, (600,), generator=g)]
    lens[0], lens[1], lens[7] = 0, unit, 64  # an empty sample first, a shortest one, a longest one
    if cp == 1 and sum(lens[:512]) % 4 == 0:  # the second group's first LSE column off a 16-byte boundary
        lens[2] += 2 if lens[2] < 64 else -2
    cu, q, k, v, do = _packed_case(lens, hq, hkv, d, seed=700 + cp)
    assert len(lens) > 512 and (cp != 1 or cu[512] % 4 != 0)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = cpattn_fwd_varlen(qd, kd, vd, cu, cp)
    dq, dk, dv = cpattn_bwd_varlen(qd, kd, vd, o, lse, dod, cu, cp)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    o_r, l_r = oracle.varlen_attention_forward(q, k, v, cu)
    err = (o.double().cpu() - o_r).abs()
    assert (err <= 1e-2 + _half_ulp_bf16(o_r)).all(), err.max().item()
    nonempty = torch.isfinite(l_r)
    assert torch.equal(torch.isfinite(lse.cpu()), nonempty)
    assert (lse.double().cpu()[nonempty] - l_r[nonempty]).abs().max().item() <= 1e-3
    dq_r, dk_r, dv_r = oracle.varlen_attention_backward(q, k, v, do, cu)
    for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
        assert _rel(got.float().cpu(), ref) <= 2e-2, name

"""Rotary position embedding (cpattn_rope) through the C ABI against the CPU
fp64 oracle (oracle/rope.py): natural order, every rank's zigzag shard,
packed samples, long positions, and the inverse rotation.

Tolerance: the output is bf16, so each element may differ from the exact
rotation of the bf16 input by half a bf16 ulp of the result plus the fp32
arithmetic (|x| * 2^-20 covers it): |got - ref| <= ulp(ref)/2 + 1e-6 * (|x1| + |x2|).
"""
import pytest
import torch

import oracle
from context_blockwise_causal_gb300 import cpattn_rope

pytestmark = pytest.mark.gpu


def _half_ulp_bf16(x):
    e = torch.floor(torch.log2(x.abs().clamp_min(2.0 ** -126)))
    return 2.0 ** (e - 8)


def _check(got, x, pos, base=10000.0, inverse=False):
    ref = oracle.rope_apply(x.double().cpu(), pos, base=base, inverse=inverse)
    got = got.double().cpu()
    d = x.shape[-1]
    mag = x.double().cpu().abs()
    pair = torch.cat([mag[..., :d // 2] + mag[..., d // 2:]] * 2, dim=-1)
    bound = _half_ulp_bf16(ref) + 1e-6 * pair + 1e-30
    assert ((got - ref).abs() <= bound).all(), ((got - ref).abs() - bound).max().item()


def _x(b, n, h, d, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(b, n, h, d, generator=g) * 2).to(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
def test_rope_natural_order(d):
    x = _x(2, 1000, 3, d, 1)
    got = cpattn_rope(x.cuda())
    torch.cuda.synchronize()
    _check(got, x, oracle.natural_positions(1000))


@pytest.mark.parametrize("cp", [1, 2, 3, 8])
def test_rope_rank_shards_use_global_positions(cp):
    s = 96 * cp
    x = _x(1, s, 4, 128, 2 + cp)
    for r in range(cp):
        idx = oracle.zigzag_global_index(s, cp)[r]
        shard = x[:, idx].contiguous()
        got = cpattn_rope(shard.cuda(), cp=cp, rank=r, s=s)
        torch.cuda.synchronize()
        _check(got, shard, oracle.rank_local_positions(s, cp, r))


def test_rope_packed_samples():
    s, cp = 1200, 3
    cu = [0, 100, 101, 640, 1200]
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    x = _x(1, s, 2, 64, 7)
    got = cpattn_rope(x.cuda(), cu_seqlens=cu_dev)
    torch.cuda.synchronize()
    _check(got, x, oracle.natural_positions(s, cu))
    for r in range(cp):
        idx = oracle.zigzag_global_index(s, cp)[r]
        shard = x[:, idx].contiguous()
        got = cpattn_rope(shard.cuda(), cp=cp, rank=r, s=s, cu_seqlens=cu_dev)
        torch.cuda.synchronize()
        _check(got, shard, oracle.rank_local_positions(s, cp, r, cu))


def test_rope_long_positions_and_base():
    s = 131072
    x = _x(1, s, 2, 128, 9)
    got = cpattn_rope(x.cuda(), base=500000.0)
    torch.cuda.synchronize()
    rows = torch.cat([torch.arange(0, 64), torch.arange(s - 4096, s)])
    _check(got[:, rows.cuda()], x[:, rows], rows, base=500000.0)


def test_rope_inverse_undoes_the_rotation():
    x = _x(2, 512, 4, 128, 11)
    y = cpattn_rope(x.cuda())
    _check(y.clone(), x, oracle.natural_positions(512))
    z = cpattn_rope(y, inverse=True)
    torch.cuda.synchronize()
    # two bf16 roundings apart from x; a rounding error of either element of
    # a pair moves both after the rotation, so bound by the pair's magnitude
    xd = x.double()
    d = xd.shape[-1]
    pm = torch.maximum(xd[..., :d // 2].abs(), xd[..., d // 2:].abs())
    pm = torch.cat([pm, pm], dim=-1)
    diff = (z.double().cpu() - xd).abs()
    assert (diff <= 4 * _half_ulp_bf16(pm) + 1e-6 * pm).all()

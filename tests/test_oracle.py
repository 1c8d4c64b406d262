"""Pins for the CPU fp64 oracle, independent of the oracle's own code.

Each pin comes from outside the oracle: hand-derived values (tests/golden),
closed forms, a library attention routine (torch's scaled_dot_product_attention
and autograd, float64), central finite differences, gradient identities, and
the agreement of the two independent routes (plain definition vs. the CP
step/merge procedure).
"""
import json
import math
import os
import random

import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import attention_backward, attention_forward, cp_attention_forward

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F64 = torch.float64


def _num(x):
    if isinstance(x, (int, float)):
        return float(x)
    table = {"ln3": math.log(3), "ln4": math.log(4), "ln5": math.log(5), "sqrt2ln2": math.sqrt(2) * math.log(2),
             "5/3": 5 / 3, "10/3": 10 / 3, "0.75ln3": 0.75 * math.log(3)}
    return table[x]


def _t(rows):
    return torch.tensor([[_num(x) for x in row] for row in rows], dtype=F64)


def _rand(*shape, gen, std=1.0):
    return torch.randn(*shape, generator=gen, dtype=F64) * std


def _library_attention(q, k, v, causal):
    """torch SDPA in float64 with K/V heads repeated for GQA: [b,s,h,d] layout."""
    G = q.shape[2] // k.shape[2]
    kk = k.repeat_interleave(G, dim=2)
    vv = v.repeat_interleave(G, dim=2)
    out = F.scaled_dot_product_attention(q.transpose(1, 2), kk.transpose(1, 2), vv.transpose(1, 2),
                                         is_causal=causal)
    return out.transpose(1, 2)


def _library_lse(q, k, causal):
    G = q.shape[2] // k.shape[2]
    kk = k.repeat_interleave(G, dim=2)
    S = torch.einsum("bthd,bjhd->bhtj", q, kk) / math.sqrt(q.shape[-1])
    if causal:
        s = q.shape[1]
        S = S.masked_fill(torch.ones(s, s, dtype=torch.bool).triu(1), float("-inf"))
    return torch.logsumexp(S, dim=-1)


# ------------------------------------------------------------ hand values
def test_golden_forward():
    data = json.load(open(os.path.join(GOLDEN, "hand_attention.json")))
    for case in data["cases"]:
        q, k, v = (_t(case[n])[None, :, None, :] for n in ("q", "k", "v"))
        for mode, causal in (("causal", True), ("full", False)):
            o, lse = attention_forward(q, k, v, causal=causal)
            want_o = _t(case[mode]["o"])
            want_l = torch.tensor([_num(x) for x in case[mode]["lse"]], dtype=F64)
            assert torch.allclose(o[0, :, 0], want_o, atol=1e-13), (case["name"], mode)
            assert torch.allclose(lse[0, 0], want_l, atol=1e-13), (case["name"], mode)


def test_golden_backward():
    data = json.load(open(os.path.join(GOLDEN, "hand_attention.json")))
    case = data["cases"][0]
    q, k, v = (_t(case[n])[None, :, None, :] for n in ("q", "k", "v"))
    bw = case["backward"]
    do = _t(bw["do"])[None, :, None, :]
    dq, dk, dv = attention_backward(q, k, v, do, causal=True)
    assert torch.allclose(dq[0, :, 0], _t(bw["dq"]), atol=1e-13)
    assert torch.allclose(dk[0, :, 0], _t(bw["dk"]), atol=1e-13)
    assert torch.allclose(dv[0, :, 0], _t(bw["dv"]), atol=1e-13)


# ------------------------------------------------------------ library routine
@pytest.mark.parametrize("b,s,hq,hkv,d", [(1, 1, 1, 1, 4), (2, 37, 4, 2, 8), (1, 50, 6, 3, 16), (1, 64, 8, 1, 5)])
@pytest.mark.parametrize("causal", [True, False])
def test_forward_matches_library(b, s, hq, hkv, d, causal):
    g = torch.Generator().manual_seed(s * 131 + hq)
    q, k, v = _rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g)
    o, lse = attention_forward(q, k, v, causal=causal, row_block=16)
    assert torch.allclose(o, _library_attention(q, k, v, causal), atol=1e-12, rtol=0)
    assert torch.allclose(lse, _library_lse(q, k, causal), atol=1e-12, rtol=0)


@pytest.mark.parametrize("b,s,hq,hkv,d", [(1, 19, 2, 1, 4), (2, 24, 4, 2, 8)])
@pytest.mark.parametrize("causal", [True, False])
def test_backward_matches_autograd(b, s, hq, hkv, d, causal):
    g = torch.Generator().manual_seed(7 + s)
    q, k, v, do = (_rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g),
                   _rand(b, s, hq, d, gen=g))
    qa, ka, va = (x.clone().requires_grad_(True) for x in (q, k, v))
    (_library_attention(qa, ka, va, causal) * do).sum().backward()
    dq, dk, dv = attention_backward(q, k, v, do, causal=causal, row_block=8)
    assert torch.allclose(dq, qa.grad, atol=1e-11, rtol=0)
    assert torch.allclose(dk, ka.grad, atol=1e-11, rtol=0)
    assert torch.allclose(dv, va.grad, atol=1e-11, rtol=0)


# ------------------------------------------------------------ closed forms / invariants
def test_zero_query_gives_running_mean():
    g = torch.Generator().manual_seed(3)
    s, d = 33, 6
    q = torch.zeros(1, s, 2, d, dtype=F64)
    k, v = _rand(1, s, 1, d, gen=g), _rand(1, s, 1, d, gen=g)
    o, lse = attention_forward(q, k, v, causal=True)
    mean = torch.cumsum(v[0, :, 0], dim=0) / torch.arange(1, s + 1, dtype=F64)[:, None]
    for h in range(2):
        assert torch.allclose(o[0, :, h], mean, atol=1e-13)
        assert torch.allclose(lse[0, h], torch.log(torch.arange(1, s + 1, dtype=F64)), atol=1e-13)


def test_constant_values_pass_through():
    g = torch.Generator().manual_seed(4)
    s, d = 20, 5
    q, k = _rand(1, s, 1, d, gen=g, std=3), _rand(1, s, 1, d, gen=g, std=3)
    row = _rand(d, gen=g)
    v = row.expand(1, s, 1, d).clone()
    o, _ = attention_forward(q, k, v, causal=True)
    assert torch.allclose(o[0, :, 0], row.expand(s, d), atol=1e-12)


def test_probability_rows_sum_to_one_and_respect_mask():
    # one-hot values expose the probability matrix itself: O[t] = P[t, :]
    g = torch.Generator().manual_seed(5)
    s = d = 12
    q, k = _rand(1, s, 1, d, gen=g, std=2), _rand(1, s, 1, d, gen=g, std=2)
    v = torch.eye(s, dtype=F64)[None, :, None, :]
    P, _ = attention_forward(q, k, v, causal=True)
    P = P[0, :, 0]
    assert torch.allclose(P.sum(dim=1), torch.ones(s, dtype=F64), atol=1e-14)
    assert torch.all(P.triu(1) == 0)
    assert torch.all(P[torch.ones(s, s, dtype=torch.bool).tril()] > 0)


def test_backward_finite_differences():
    g = torch.Generator().manual_seed(11)
    b, s, hq, hkv, d = 1, 6, 2, 1, 3
    q, k, v, do = (_rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g),
                   _rand(b, s, hq, d, gen=g))

    def loss(q_, k_, v_):
        return float((attention_forward(q_, k_, v_, causal=True)[0] * do).sum())

    dq, dk, dv = attention_backward(q, k, v, do, causal=True)
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = torch.zeros_like(x)
        flat, nflat = x.view(-1), num.view(-1)
        for i in range(flat.numel()):
            old = float(flat[i])
            flat[i] = old + eps
            up = loss(q, k, v)
            flat[i] = old - eps
            dn = loss(q, k, v)
            flat[i] = old
            nflat[i] = (up - dn) / (2 * eps)
        assert torch.allclose(grad, num, atol=1e-7, rtol=1e-6), name


def test_gradient_identities():
    g = torch.Generator().manual_seed(12)
    b, s, hq, hkv, d = 2, 29, 4, 2, 8
    q, k, v, do = (_rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g),
                   _rand(b, s, hq, d, gen=g))
    _, dk, dv = attention_backward(q, k, v, do, causal=True, row_block=7)
    G = hq // hkv
    # rows of P sum to 1  =>  sum_j dV_j = sum over the group's heads and all t of dO_t
    want = do.view(b, s, hkv, G, d).sum(dim=(1, 3))
    assert torch.allclose(dv.sum(dim=1), want, atol=1e-12)
    # rows of dS sum to 0  =>  sum_j dK_j = 0
    assert torch.allclose(dk.sum(dim=1), torch.zeros_like(want), atol=1e-12)


def test_row_and_head_subsets_match_full():
    g = torch.Generator().manual_seed(13)
    b, s, hq, hkv, d = 1, 40, 4, 2, 8
    q, k, v, do = (_rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g),
                   _rand(b, s, hq, d, gen=g))
    rows = [39, 0, 17, 5]
    o_full, l_full = attention_forward(q, k, v)
    o_s, l_s = attention_forward(q, k, v, rows=rows)
    assert torch.equal(o_s, o_full[:, rows]) or torch.allclose(o_s, o_full[:, rows], atol=1e-14)
    assert torch.allclose(l_s, l_full[:, :, rows], atol=1e-14)
    dq_f, dk_f, dv_f = attention_backward(q, k, v, do)
    dq_s, dk_s, dv_s = attention_backward(q, k, v, do, dq_rows=rows, dkv_heads=[1])
    assert torch.allclose(dq_s, dq_f[:, rows], atol=1e-13)
    assert torch.allclose(dk_s[:, :, 0], dk_f[:, :, 1], atol=1e-13)
    assert torch.allclose(dv_s[:, :, 0], dv_f[:, :, 1], atol=1e-13)


# ------------------------------------------------------------ the CP route
def test_zigzag_split_golden():
    data = json.load(open(os.path.join(GOLDEN, "zigzag_split.json")))
    for case in data["cases"]:
        if "chunks" in case:
            assert [list(ch) for _, ch in oracle.zigzag_chunks(case["cp"])] == case["chunks"]
        else:
            got = oracle.zigzag_global_index(case["s"], case["cp"]).tolist()
            assert got == case["global_of_local"]


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 5, 8, 16])
def test_zigzag_index_is_a_balanced_bijection(cp):
    c = 3
    s = 2 * cp * c
    idx = oracle.zigzag_global_index(s, cp)
    assert sorted(idx.reshape(-1).tolist()) == list(range(s))
    # each rank's causal work (number of visible keys) is the same
    work = [(idx[r] + 1).sum().item() for r in range(cp)]
    assert len(set(work)) == 1


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 6])
@pytest.mark.parametrize("causal", [True, False])
def test_step_plan_covers_each_pair_once(cp, causal):
    """Brute force: the blocks of every rank's steps cover each visible
    (query, key) pair of its rows exactly once, and no masked pair except
    inside the causal step."""
    c = 2
    s = 2 * cp * c
    for r in range(cp):
        count = torch.zeros(s, s, dtype=torch.long)
        for (_i, _j, q_ch, kv_ch, masked) in oracle.cp_step_plan(r, cp, causal):
            for qc in q_ch:
                for kc in kv_ch:
                    for t in range(qc * c, (qc + 1) * c):
                        for j in range(kc * c, (kc + 1) * c):
                            if masked and j > t:
                                continue
                            assert not causal or j <= t, "unmasked block reaches a future key"
                            count[t, j] += 1
        mine = oracle.zigzag_global_index(s, cp)[r].tolist()
        for t in range(s):
            want = [1 if (t in mine and (j <= t or not causal)) else 0 for j in range(s)]
            assert count[t].tolist() == want, (r, t)


@pytest.mark.parametrize("b,s,hq,hkv,d,cp", [(1, 8, 1, 1, 4, 1), (1, 24, 2, 1, 4, 3), (2, 32, 4, 2, 8, 4),
                                              (1, 40, 2, 2, 3, 5)])
@pytest.mark.parametrize("causal", [True, False])
def test_cp_route_equals_uncut(b, s, hq, hkv, d, cp, causal):
    g = torch.Generator().manual_seed(100 + s + cp)
    q, k, v = _rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g)
    o_ref, l_ref = attention_forward(q, k, v, causal=causal)
    o_cp, l_cp = cp_attention_forward(q, k, v, cp, causal=causal)
    assert torch.allclose(o_cp, o_ref, atol=1e-12, rtol=0)
    assert torch.allclose(l_cp, l_ref, atol=1e-12, rtol=0)


def test_merge_is_order_independent():
    g = torch.Generator().manual_seed(21)
    b, s, hq, hkv, d, cp = 1, 32, 2, 1, 8, 4
    q, k, v = _rand(b, s, hq, d, gen=g, std=2), _rand(b, s, hkv, d, gen=g, std=2), _rand(b, s, hkv, d, gen=g)
    o0, l0 = cp_attention_forward(q, k, v, cp)
    rng = random.Random(5)

    def shuffled(idx):
        idx = list(idx)
        rng.shuffle(idx)
        return idx

    for order in (lambda x: list(reversed(x)), shuffled, shuffled):
        o1, l1 = cp_attention_forward(q, k, v, cp, merge_order=order)
        assert torch.allclose(o1, o0, atol=1e-12)
        assert torch.allclose(l1, l0, atol=1e-12)


def test_lse_merge_two_halves_closed_form():
    # exp(L) of the merge is the sum of the parts' exp(L): log-add-exp by hand
    L1, L2 = torch.tensor([0.0, 2.0], dtype=F64), torch.tensor([math.log(3.0), -1.0], dtype=F64)
    O1, O2 = torch.tensor([[1.0], [0.0]], dtype=F64), torch.tensor([[5.0], [4.0]], dtype=F64)
    O, L = oracle.lse_merge([(O1, L1), (O2, L2)])
    assert abs(L[0] - math.log(4.0)) < 1e-15
    assert abs(O[0, 0] - (1.0 * 1 / 4 + 5.0 * 3 / 4)) < 1e-14
    w = 1.0 / (1.0 + math.exp(-3.0))
    assert abs(L[1] - (2.0 + math.log(1 + math.exp(-3.0)))) < 1e-14
    assert abs(O[1, 0] - 4.0 * (1 - w)) < 1e-14


@pytest.mark.parametrize("b,s,hq,hkv,d,cp,causal", [(1, 24, 2, 1, 4, 3, True), (2, 32, 4, 2, 8, 4, True),
                                                    (1, 40, 2, 2, 3, 5, True), (1, 24, 2, 2, 4, 3, False)])
def test_step_partials_merge_to_uncut(b, s, hq, hkv, d, cp, causal):
    """Merging the cp per-step partials row by row gives uncut attention."""
    g = torch.Generator().manual_seed(300 + s + cp)
    q, k, v = _rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g)
    o_ref, l_ref = attention_forward(q, k, v, causal=causal)
    parts = [oracle.cp_step_partials(q, k, v, cp, i, causal=causal) for i in range(cp)]
    for bi in range(b):
        for h in range(hq):
            O, L = oracle.lse_merge([(o_i[bi, :, h], l_i[bi, h]) for o_i, l_i in parts])
            assert torch.allclose(O, o_ref[bi, :, h], atol=1e-12, rtol=0)
            assert torch.allclose(L, l_ref[bi, h], atol=1e-12, rtol=0)


def test_step_partials_structure():
    """Which rows take part in each step ([MLM-CP] 3.4), and step 0 of the
    first chunk being plain causal attention over that chunk's prefix."""
    b, s, hq, hkv, d, cp = 1, 32, 2, 1, 4, 4
    c = s // (2 * cp)
    g = torch.Generator().manual_seed(7)
    q, k, v = _rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g)
    o_ref, l_ref = attention_forward(q, k, v)
    for i in range(cp):
        o_i, l_i = oracle.cp_step_partials(q, k, v, cp, i)
        for r in range(cp):
            lo, hi = range(r * c, (r + 1) * c), range((2 * cp - 1 - r) * c, (2 * cp - r) * c)
            first_in = i <= r  # the first chunk's rows take part in steps 0..r
            assert bool(torch.isfinite(l_i[0, :, list(lo)]).all()) == first_in
            assert torch.isfinite(l_i[0, :, list(hi)]).all()  # the second chunk's rows in every step
            if not first_in:
                assert (o_i[0, list(lo)] == 0).all()
        if i == 0:
            # chunk 0 (rank 0's first chunk) sees exactly keys 0..t at step 0
            assert torch.allclose(o_i[0, :c], o_ref[0, :c], atol=1e-12)
            assert torch.allclose(l_i[0, :, :c], l_ref[0, :, :c], atol=1e-12)


# ---------------------------------------------------------------- RoPE
def test_rope_hand_values():
    # d = 2, base irrelevant for i = 0: a plain rotation by pos radians
    x = torch.tensor([[[[1.0, 0.0]], [[1.0, 0.0]], [[0.0, 2.0]]]], dtype=F64)  # [1, 3, 1, 2]
    out = oracle.rope_apply(x, torch.tensor([0, 1, 3]))
    assert torch.allclose(out[0, 0, 0], torch.tensor([1.0, 0.0], dtype=F64), atol=0)
    assert torch.allclose(out[0, 1, 0], torch.tensor([math.cos(1.0), math.sin(1.0)], dtype=F64), atol=1e-15)
    assert torch.allclose(out[0, 2, 0], torch.tensor([-2 * math.sin(3.0), 2 * math.cos(3.0)], dtype=F64), atol=1e-15)
    # d = 4: the second pair turns base^(-1/2) as fast
    th = oracle.rope_angles(torch.tensor([5]), 4, base=100.0)
    assert abs(th[0, 0] - 5.0) < 1e-15 and abs(th[0, 1] - 0.5) < 1e-15


def test_rope_relative_phase_and_inverse():
    g = torch.Generator().manual_seed(3)
    d = 16
    q, k = torch.randn(1, 1, 1, d, generator=g, dtype=F64), torch.randn(1, 1, 1, d, generator=g, dtype=F64)
    dots = []
    for m, n in ((7, 3), (104, 100), (4, 0)):  # m - n = 4 each time
        qm = oracle.rope_apply(q, torch.tensor([m]))
        kn = oracle.rope_apply(k, torch.tensor([n]))
        dots.append(float((qm * kn).sum()))
    assert max(dots) - min(dots) < 1e-12
    x = torch.randn(2, 5, 3, d, generator=g, dtype=F64)
    pos = torch.tensor([0, 9, 33, 1000, 131071])
    y = oracle.rope_apply(x, pos)
    # pair norms are kept, the inverse undoes the rotation
    assert torch.allclose(y[..., :d // 2] ** 2 + y[..., d // 2:] ** 2, x[..., :d // 2] ** 2 + x[..., d // 2:] ** 2,
                          atol=1e-12)
    assert torch.allclose(oracle.rope_apply(y, pos, inverse=True), x, atol=1e-12)


def test_rope_positions_for_cp_shards_and_packing():
    s, cp = 48, 3
    c = s // (2 * cp)
    # rank-local positions are the zigzag global positions, not 0..2c-1
    for r in range(cp):
        pos = oracle.rank_local_positions(s, cp, r)
        assert pos.tolist() == list(range(r * c, (r + 1) * c)) + list(range((2 * cp - 1 - r) * c, (2 * cp - r) * c))
    # packing: the position restarts at each sample
    cu = [0, 10, 30, 48]
    pos = oracle.natural_positions(s, cu)
    assert pos.tolist() == list(range(10)) + list(range(20)) + list(range(18))
    # rotating a rank's shard with its local positions = rotating the whole
    # sequence and taking the shard
    g = torch.Generator().manual_seed(4)
    x = torch.randn(1, s, 2, 8, generator=g, dtype=F64)
    full = oracle.rope_apply(x, oracle.natural_positions(s, cu))
    for r in range(cp):
        idx = oracle.zigzag_global_index(s, cp)[r]
        shard = oracle.rope_apply(x[:, idx], oracle.rank_local_positions(s, cp, r, cu))
        assert torch.allclose(shard, full[:, idx], atol=1e-15)


# ---------------------------------------------------------------- user scale
def test_scale_zero_gives_uniform_weights():
    # scale 0: every visible key weighs the same: O = running mean of v, L = log(t+1)
    g = torch.Generator().manual_seed(12)
    q, k, v = _rand(1, 6, 1, 4, gen=g), _rand(1, 6, 1, 4, gen=g), _rand(1, 6, 1, 4, gen=g)
    o, lse = attention_forward(q, k, v, scale=0.0)
    for t in range(6):
        assert torch.allclose(o[0, t, 0], v[0, :t + 1, 0].mean(dim=0), atol=1e-14)
        assert abs(lse[0, 0, t] - math.log(t + 1)) < 1e-14


def test_scale_moves_into_the_queries():
    # scale * (q . k) = (alpha q) . k * (scale / alpha): forward and gradients
    g = torch.Generator().manual_seed(13)
    b, s, hq, hkv, d = 1, 12, 2, 1, 8
    q, k, v, do = (_rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g),
                   _rand(b, s, hq, d, gen=g))
    alpha, sc = 3.0, 0.7
    o1, l1 = attention_forward(q, k, v, scale=sc)
    o2, l2 = attention_forward(q * alpha, k, v, scale=sc / alpha)
    assert torch.allclose(o1, o2, atol=1e-12) and torch.allclose(l1, l2, atol=1e-12)
    dq1, dk1, dv1 = attention_backward(q, k, v, do, scale=sc)
    dq2, dk2, dv2 = attention_backward(q * alpha, k, v, do, scale=sc / alpha)
    assert torch.allclose(dq1, dq2 * alpha, atol=1e-12)
    assert torch.allclose(dk1, dk2, atol=1e-12) and torch.allclose(dv1, dv2, atol=1e-12)
    # default is 1/sqrt(d)
    o3, _ = attention_forward(q, k, v, scale=1 / math.sqrt(d))
    o4, _ = attention_forward(q, k, v)
    assert torch.equal(o3, o4)


# ---------------------------------------------------------------- packed samples
def test_varlen_uniform_lengths_equal_a_batch():
    g = torch.Generator().manual_seed(14)
    b, L, hq, hkv, d = 3, 10, 2, 1, 4
    q, k, v, do = (_rand(b, L, hq, d, gen=g), _rand(b, L, hkv, d, gen=g), _rand(b, L, hkv, d, gen=g),
                   _rand(b, L, hq, d, gen=g))
    o, lse = attention_forward(q, k, v)
    cu = [0, L, 2 * L, 3 * L]
    flat = lambda t: t.reshape(b * L, t.shape[2], t.shape[3])  # noqa: E731
    ov, lv = oracle.varlen_attention_forward(flat(q), flat(k), flat(v), cu)
    assert torch.allclose(ov, flat(o), atol=1e-14)
    assert torch.allclose(lv, lse.permute(1, 0, 2).reshape(hq, b * L), atol=1e-14)
    dq, dk, dv = attention_backward(q, k, v, do)
    gq, gk, gv = oracle.varlen_attention_backward(flat(q), flat(k), flat(v), flat(do), cu)
    assert torch.allclose(gq, flat(dq), atol=1e-13) and torch.allclose(gk, flat(dk), atol=1e-13)
    assert torch.allclose(gv, flat(dv), atol=1e-13)


def test_varlen_samples_do_not_see_each_other():
    g = torch.Generator().manual_seed(15)
    total, hq, hkv, d = 20, 2, 2, 4
    cu = [0, 6, 6, 20]  # an empty sample in the middle
    q, k, v = _rand(1, total, hq, d, gen=g)[0], _rand(1, total, hkv, d, gen=g)[0], _rand(1, total, hkv, d, gen=g)[0]
    o1, l1 = oracle.varlen_attention_forward(q, k, v, cu)
    k2, v2 = k.clone(), v.clone()
    k2[6:] += 1.0
    v2[6:] -= 2.0
    o2, l2 = oracle.varlen_attention_forward(q, k2, v2, cu)
    assert torch.equal(o1[:6], o2[:6]) and torch.equal(l1[:, :6], l2[:, :6])
    # the first token of the second sample attends only to itself: O = v, L = scale q.k
    assert torch.allclose(o1[6], v[6].to(F64).repeat_interleave(hq // hkv, dim=0), atol=1e-14)
    sc = 1 / math.sqrt(d)
    assert torch.allclose(l1[:, 6], (q[6].to(F64) * k[6].to(F64)).sum(-1) * sc, atol=1e-14)

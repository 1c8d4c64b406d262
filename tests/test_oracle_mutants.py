"""The oracle's pins catch planted mistakes.

Each mutant is a copy of the ``oracle`` package with one plausible mistake
written into its source (a dropped term, a wrong sign, index or operand, an
off-by-one mask, a wrong log base, ...). The pins below come from outside the
oracle -- hand-derived golden values (tests/golden), torch's float64 SDPA and
autograd, closed forms -- and every mutant must fail at least one of them,
while the unmodified copy passes them all. Everything runs on the CPU.
"""
import importlib
import json
import math
import os
import shutil
import sys

import pytest
import torch
import torch.nn.functional as F

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_DIR = os.path.join(os.path.dirname(HERE), "oracle")
GOLDEN = os.path.join(HERE, "golden")
F64 = torch.float64


# ---------------------------------------------------------------- references
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


def _sdpa(q, k, v, causal):
    G = q.shape[2] // k.shape[2]
    kk, vv = k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2)
    out = F.scaled_dot_product_attention(q.transpose(1, 2), kk.transpose(1, 2), vv.transpose(1, 2), is_causal=causal)
    return out.transpose(1, 2)


def _lse(q, k, causal):
    G = q.shape[2] // k.shape[2]
    S = torch.einsum("bthd,bjhd->bhtj", q, k.repeat_interleave(G, dim=2)) / math.sqrt(q.shape[-1])
    if causal:
        s = q.shape[1]
        S = S.masked_fill(torch.ones(s, s, dtype=torch.bool).triu(1), float("-inf"))
    return torch.logsumexp(S, dim=-1)


def _close(a, b, tol):
    assert torch.allclose(a, b, atol=tol, rtol=0), float((a - b).abs().max())


# ---------------------------------------------------------------- pins
def pin_golden_forward(M):
    for case in json.load(open(os.path.join(GOLDEN, "hand_attention.json")))["cases"]:
        q, k, v = (_t(case[n])[None, :, None, :] for n in ("q", "k", "v"))
        for mode, causal in (("causal", True), ("full", False)):
            o, lse = M.attention_forward(q, k, v, causal=causal)
            _close(o[0, :, 0], _t(case[mode]["o"]), 1e-12)
            _close(lse[0, 0], torch.tensor([_num(x) for x in case[mode]["lse"]], dtype=F64), 1e-12)


def pin_golden_backward(M):
    case = json.load(open(os.path.join(GOLDEN, "hand_attention.json")))["cases"][0]
    q, k, v = (_t(case[n])[None, :, None, :] for n in ("q", "k", "v"))
    bw = case["backward"]
    dq, dk, dv = M.attention_backward(q, k, v, _t(bw["do"])[None, :, None, :], causal=True)
    for got, key in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _close(got[0, :, 0], _t(bw[key]), 1e-12)


SHAPES = [(2, 21, 4, 2, 8), (1, 16, 6, 3, 5), (1, 12, 2, 2, 4)]


def pin_forward_library(M):
    for i, (b, s, hq, hkv, d) in enumerate(SHAPES):
        g = torch.Generator().manual_seed(40 + i)
        q, k, v = _rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g)
        for causal in (True, False):
            o, lse = M.attention_forward(q, k, v, causal=causal, row_block=8)
            _close(o, _sdpa(q, k, v, causal), 1e-11)
            _close(lse, _lse(q, k, causal), 1e-11)


def pin_backward_autograd(M):
    for i, (b, s, hq, hkv, d) in enumerate(SHAPES):
        g = torch.Generator().manual_seed(60 + i)
        q, k, v, do = (_rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g),
                       _rand(b, s, hq, d, gen=g))
        for causal in (True, False):
            qa, ka, va = (x.clone().requires_grad_(True) for x in (q, k, v))
            (_sdpa(qa, ka, va, causal) * do).sum().backward()
            dq, dk, dv = M.attention_backward(q, k, v, do, causal=causal, row_block=8)
            _close(dq, qa.grad, 1e-10)
            _close(dk, ka.grad, 1e-10)
            _close(dv, va.grad, 1e-10)


CP_CASES = [(1, 24, 2, 1, 4, 3), (2, 32, 4, 2, 8, 4), (1, 40, 2, 2, 3, 5)]


def pin_cp_route(M):
    for i, (b, s, hq, hkv, d, cp) in enumerate(CP_CASES):
        g = torch.Generator().manual_seed(80 + i)
        q, k, v = _rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g)
        for causal in (True, False):
            o, lse = M.cp_attention_forward(q, k, v, cp, causal=causal)
            _close(o, _sdpa(q, k, v, causal), 1e-11)
            _close(lse, _lse(q, k, causal), 1e-11)


def pin_step_partials(M):
    b, s, hq, hkv, d, cp = 1, 24, 2, 1, 4, 3
    g = torch.Generator().manual_seed(90)
    q, k, v = _rand(b, s, hq, d, gen=g), _rand(b, s, hkv, d, gen=g), _rand(b, s, hkv, d, gen=g)
    parts = [M.cp_step_partials(q, k, v, cp, i, causal=True) for i in range(cp)]
    o_ref, l_ref = _sdpa(q, k, v, True), _lse(q, k, True)
    for h in range(hq):
        o, lse = M.lse_merge([(p[0][0, :, h], p[1][0, h]) for p in parts])
        _close(o, o_ref[0, :, h], 1e-11)
        _close(lse, l_ref[0, h], 1e-11)


def pin_merge_closed_form(M):
    L1, L2 = torch.tensor([0.0, 2.0], dtype=F64), torch.tensor([math.log(3.0), -1.0], dtype=F64)
    O1, O2 = torch.tensor([[1.0], [0.0]], dtype=F64), torch.tensor([[5.0], [4.0]], dtype=F64)
    O, L = M.lse_merge([(O1, L1), (O2, L2)])
    w = 1.0 / (1.0 + math.exp(-3.0))
    want_L = torch.tensor([math.log(4.0), 2.0 + math.log(1 + math.exp(-3.0))], dtype=F64)
    want_O = torch.tensor([[0.25 + 5.0 * 0.75], [4.0 * (1 - w)]], dtype=F64)
    _close(L, want_L, 1e-14)
    _close(O, want_O, 1e-14)


def pin_zigzag(M):
    for case in json.load(open(os.path.join(GOLDEN, "zigzag_split.json")))["cases"]:
        if "chunks" in case:
            assert [list(ch) for _, ch in M.zigzag_chunks(case["cp"])] == case["chunks"]
        else:
            assert M.zigzag_global_index(case["s"], case["cp"]).tolist() == case["global_of_local"]


def pin_rope(M):
    x = torch.tensor([[[[1.0, 0.0]], [[1.0, 0.0]], [[0.0, 2.0]]]], dtype=F64)
    out = M.rope_apply(x, torch.tensor([0, 1, 3]))
    _close(out[0, 1, 0], torch.tensor([math.cos(1.0), math.sin(1.0)], dtype=F64), 1e-15)
    _close(out[0, 2, 0], torch.tensor([-2 * math.sin(3.0), 2 * math.cos(3.0)], dtype=F64), 1e-15)
    th = M.rope_angles(torch.tensor([5]), 4, base=100.0)
    _close(th[0], torch.tensor([5.0, 0.5], dtype=F64), 1e-15)
    s, cp = 48, 3
    c = s // (2 * cp)
    for r in range(cp):
        want = list(range(r * c, (r + 1) * c)) + list(range((2 * cp - 1 - r) * c, (2 * cp - r) * c))
        assert M.rank_local_positions(s, cp, r).tolist() == want
    assert M.natural_positions(s, [0, 10, 30, 48]).tolist() == list(range(10)) + list(range(20)) + list(range(18))


def pin_varlen(M):
    g = torch.Generator().manual_seed(95)
    lens, hq, hkv, d = [5, 9, 6], 2, 1, 4
    total = sum(lens)
    q, k, v = _rand(total, hq, d, gen=g), _rand(total, hkv, d, gen=g), _rand(total, hkv, d, gen=g)
    cu = [0, 5, 14, 20]
    for causal in (True, False):
        o, lse = M.varlen_attention_forward(q, k, v, cu, causal=causal)
        for i in range(len(lens)):
            sl = slice(cu[i], cu[i + 1])
            _close(o[sl], _sdpa(q[None, sl], k[None, sl], v[None, sl], causal)[0], 1e-11)
            _close(lse[:, sl], _lse(q[None, sl], k[None, sl], causal)[0], 1e-11)


def pin_varlen_backward(M):
    g = torch.Generator().manual_seed(96)
    hq, hkv, d, cu = 2, 1, 4, [0, 6, 6, 13]
    total = cu[-1]
    q, k, v, do = (_rand(total, hq, d, gen=g), _rand(total, hkv, d, gen=g), _rand(total, hkv, d, gen=g),
                   _rand(total, hq, d, gen=g))
    dq, dk, dv = M.varlen_attention_backward(q, k, v, do, cu, causal=True)
    for a, b in ((0, 6), (6, 13)):
        qa, ka, va = (x[None, a:b].clone().requires_grad_(True) for x in (q, k, v))
        (_sdpa(qa, ka, va, True) * do[None, a:b]).sum().backward()
        _close(dq[a:b], qa.grad[0], 1e-10)
        _close(dk[a:b], ka.grad[0], 1e-10)
        _close(dv[a:b], va.grad[0], 1e-10)


PINS = [pin_golden_forward, pin_golden_backward, pin_forward_library, pin_backward_autograd, pin_cp_route,
        pin_step_partials, pin_merge_closed_form, pin_zigzag, pin_rope, pin_varlen, pin_varlen_backward]


# ---------------------------------------------------------------- mutants
# (name, file, text in the oracle, its replacement)
MUTANTS = [
    ("mask_excludes_diagonal", "attention.py", "S.masked_fill_(j[None, :] > t[:, None]", "S.masked_fill_(j[None, :] >= t[:, None]"),
    ("scale_one_over_d", "attention.py", "return 1.0 / math.sqrt(d)", "return 1.0 / d"),
    ("lse_log2", "attention.py", "L = m_safe + torch.log(torch.exp(S - m_safe)", "L = m_safe + torch.log2(torch.exp(S - m_safe)"),
    ("output_uses_keys", "attention.py", "o[bi, r0:r0 + t.numel(), h] = P @ vv_all[:nk]", "o[bi, r0:r0 + t.numel(), h] = P @ kk_all[:nk]"),
    ("gqa_interleaved_forward", "attention.py",
     "            vv_all = v[bi, :, g].to(_F64)\n            for h in range(g * G, (g + 1) * G):",
     "            vv_all = v[bi, :, g].to(_F64)\n            for h in range(g, hq, hkv):"),
    ("dS_drops_row_term", "attention.py", "dS = P * (dP - (P * dP).sum(dim=1, keepdim=True))", "dS = P * dP"),
    ("dS_sign", "attention.py", "dS = P * (dP - (P * dP).sum(dim=1, keepdim=True))", "dS = P * ((P * dP).sum(dim=1, keepdim=True) - dP)"),
    ("dK_without_scale", "attention.py", "dk[bi, :nk, slot] += scale * (dS.T @ qq)", "dk[bi, :nk, slot] += dS.T @ qq"),
    ("dV_wrong_operand", "attention.py", "dv[bi, :nk, slot] += P.T @ dd", "dv[bi, :nk, slot] += P.T @ qq"),
    ("dQ_uses_values", "attention.py", "dq[bi, r0:r0 + t.numel(), h] = scale * (dS @ kk[:nk])", "dq[bi, r0:r0 + t.numel(), h] = scale * (dS @ vv[:nk])"),
    ("dP_transposed_values", "attention.py", "dP = dd @ vv[:nk].T", "dP = dd @ kk[:nk].T"),
    ("zigzag_partner_off_by_one", "context_parallel.py", "return [(r, (r, 2 * cp - 1 - r)) for r in range(cp)]",
     "return [(r, (r, 2 * cp - 2 - r if r < cp - 1 else cp)) for r in range(cp)]"),
    ("ring_direction_reversed", "context_parallel.py", "        j = (r - i) % cp\n", "        j = (r + i) % cp\n"),
    ("early_steps_take_second_half", "context_parallel.py", "plan.append((i, j, (lo, hi), (j_lo,), False))", "plan.append((i, j, (lo, hi), (j_hi,), False))"),
    ("late_steps_keep_first_q_half", "context_parallel.py", "plan.append((i, j, (hi,), (j_lo, j_hi), False))", "plan.append((i, j, (lo,), (j_lo, j_hi), False))"),
    ("step0_unmasked", "context_parallel.py", "plan.append((i, j, (lo, hi), (lo, hi), True))", "plan.append((i, j, (lo, hi), (lo, hi), False))"),
    ("block_mask_excludes_diagonal", "context_parallel.py", "S = S.masked_fill(k_pos[None, :] > q_pos[:, None]", "S = S.masked_fill(k_pos[None, :] >= q_pos[:, None]"),
    ("merge_drops_a_part", "context_parallel.py", "torch.log(torch.exp(L - m_safe) + torch.exp(Li - m_safe))", "torch.log(torch.exp(L - m_safe))"),
    ("merge_weight_sign", "context_parallel.py", "torch.exp(Li - torch.where(torch.isfinite(L), L, torch.zeros_like(L)))",
     "torch.exp(torch.where(torch.isfinite(L), L, torch.zeros_like(L)) - Li)"),
    ("rope_rotation_sign", "rope.py", "out[bi, :, :, :half] = x1 * c - x2 * s", "out[bi, :, :, :half] = x1 * c + x2 * s"),
    ("rope_frequency_exponent", "rope.py", "inv_freq = base ** (-2.0 * i / d)", "inv_freq = base ** (-1.0 * i / d)"),
    ("rope_shard_local_positions", "rope.py", "return natural_positions(s, cu_seqlens)[g]", "return natural_positions(s, cu_seqlens)[: g.numel()]"),
    ("varlen_samples_from_zero", "varlen.py", "return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]",
     "return [(cu[0], cu[i + 1]) for i in range(len(cu) - 1)]"),
    ("varlen_always_causal", "varlen.py", "oi, li = attention_forward(q[None, a:b], k[None, a:b], v[None, a:b], causal=causal, scale=scale)",
     "oi, li = attention_forward(q[None, a:b], k[None, a:b], v[None, a:b], causal=True, scale=scale)"),
    ("varlen_dk_dv_swapped", "varlen.py", "dq[a:b], dk[a:b], dv[a:b] = gq[0], gk[0], gv[0]", "dq[a:b], dk[a:b], dv[a:b] = gq[0], gv[0], gk[0]"),
]


def _load_copy(tmp_path, tag, edit=None):
    pkg = f"oracle_copy_{tag}"
    dst = tmp_path / pkg
    shutil.copytree(ORACLE_DIR, dst, ignore=shutil.ignore_patterns("__pycache__"))
    if edit is not None:
        fname, old, new = edit
        p = dst / fname
        src = p.read_text()
        assert src.count(old) == 1, f"mutation site not unique in {fname}: {old!r}"
        p.write_text(src.replace(old, new))
    sys.path.insert(0, str(tmp_path))
    try:
        return importlib.import_module(pkg)
    finally:
        sys.path.remove(str(tmp_path))


def _failures(M):
    failed = []
    for pin in PINS:
        try:
            pin(M)
        except Exception as e:  # an assertion, or the mutant breaking outright
            failed.append(f"{pin.__name__}: {type(e).__name__}")
    return failed


def test_unmodified_copy_passes_every_pin(tmp_path):
    assert _failures(_load_copy(tmp_path, "clean")) == []


@pytest.mark.parametrize("name,fname,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, fname, old, new):
    M = _load_copy(tmp_path, name, (fname, old, new))
    assert _failures(M), f"no pin catches the mutant {name}"

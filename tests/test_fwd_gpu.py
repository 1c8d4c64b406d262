"""Forward parity: the CUDA path (through the C-ABI) against the CPU fp64 oracle.

Tolerances: max |O error| <= 1e-2 and max |LSE error| <= 1e-3 for bf16
inputs with fp32 accumulation (the stated bar for this method's kernels).
O is returned in bf16, whose own rounding is half an ulp (|O| * 2^-9, more
than 1e-2 once |O| > 5.12); the bar is read as a bound on the error of the
computation on top of that unavoidable output rounding:
|O_gpu - O_ref| <= 1e-2 + ulp_bf16(O_ref) / 2, element-wise.
Small cases compare every element; the full-size workloads compare every
head at seeded random query rows, in the launch configuration bench.py uses.
"""
import pytest
import torch

import oracle
from context_blockwise_causal_gb300 import cpattn_device_status, cpattn_fwd, cpattn_fwd_step, cpattn_lse_merge
from context_blockwise_causal_gb300.workloads import WORKLOADS, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


def _bf16_half_ulp(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = x.abs()
    e = torch.floor(torch.log2(torch.where(ax > 0, ax, torch.ones_like(ax))))
    return torch.where(ax > 0, torch.exp2(e - 8), torch.zeros_like(ax))


def _check(o, lse, o_ref, lse_ref, rows=None, name="case"):
    o_gpu = o.float().cpu().double()
    l_gpu = lse.cpu().double()
    if rows is not None:
        o_gpu = o_gpu[:, rows]
        l_gpu = l_gpu[:, :, rows]
    assert torch.isfinite(o_gpu).all() and torch.isfinite(l_gpu).all()
    err = (o_gpu - o_ref).abs()
    half_ulp = _bf16_half_ulp(o_ref)
    o_err = (err - half_ulp).max().item()
    l_err = (l_gpu - lse_ref).abs().max().item()
    # the raw error and the largest half ulp are printed (pytest -s) so the
    # share of the allowance a case uses can be read off
    print(f"PARITY {name}: max|O err| raw {err.max().item():.3e}, beyond half ulp {o_err:.3e}, "
          f"max half ulp {half_ulp.max().item():.3e}, max|O_ref| {o_ref.abs().max().item():.3f}, "
          f"max|LSE err| {l_err:.3e}")
    assert o_err <= O_TOL, f"max |O err| beyond output rounding {o_err:.3e} (raw {err.max().item():.3e})"
    assert l_err <= LSE_TOL, f"max |LSE err| {l_err:.3e}"
    return o_err, l_err


def _fp32_o_by_steps(q, k, v, cp, causal):
    """The forward's O in fp32, before any bf16 rounding: the same kernel in
    its step form (one launch per CP step, normalised fp32 partials) merged
    step after step by the log-sum-exp kernel into an fp32 result."""
    b, s, hq, d = q.shape
    o_acc, l_acc = cpattn_fwd_step(q, k, v, cp, 0, causal=causal)
    if cp > 1:
        o_part = torch.empty_like(o_acc)
        l_part = torch.empty_like(l_acc)
        for i in range(1, cp):
            cpattn_fwd_step(q, k, v, cp, i, causal=causal, o_part=o_part, lse_part=l_part)
            cpattn_lse_merge(o_acc, l_acc, o_part, l_part, o_out=o_acc, lse_out=l_acc)
        del o_part, l_part
    return o_acc, l_acc


SMALL = [
    # b, s, hq, hkv, d, cp, causal   (c = s / 2cp; several tiles, ragged tails)
    (1, 256, 2, 2, 128, 1, True),     # one virtual rank, c = 128
    (1, 512, 4, 4, 64, 2, True),      # d = 64, c = 128
    (2, 1024, 4, 2, 128, 2, True),    # GQA, 2 tiles per chunk, batch 2
    (1, 960, 6, 2, 128, 3, True),     # c = 160: ragged tiles; G = 3 pairs straddle groups
    (1, 640, 3, 1, 64, 2, True),      # odd hq (last pair repeats a head), c = 160
    (1, 1536, 8, 1, 128, 4, True),    # MQA, c = 192
    (1, 96, 2, 2, 128, 3, True),      # c = 16: tiles mostly outside their chunk
    (1, 2048, 4, 4, 128, 8, True),    # many ranks, c = 128
    (1, 768, 4, 4, 128, 3, False),    # no mask
    (2, 384, 2, 1, 64, 1, False),     # no mask, cp = 1, c = 192
    (3, 8, 2, 1, 128, 4, True),       # c = 1: one token per half-chunk, batch 3
    (1, 2, 1, 1, 64, 1, True),        # the smallest case: s = 2, one head
    (1, 6, 3, 3, 64, 3, False),       # c = 1, no mask, odd hq
    (2, 2048, 4, 4, 128, 2, True),    # MHA, c = 512: units pair two query tiles of one head
    (1, 1024, 3, 1, 64, 2, False),    # tile pairs without the mask, G = 3
    (1, 1280, 2, 2, 128, 2, True),    # tile pairs, c = 320: ragged second tile of each last pair
]


@pytest.mark.parametrize("b,s,hq,hkv,d,cp,causal", SMALL)
def test_fwd_small_all_elements(b, s, hq, hkv, d, cp, causal):
    w = Workload("case", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, causal=causal, seed=7 + s + hq)
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], cp, causal=causal)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    o_ref, l_ref = oracle.attention_forward(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), causal=causal)
    _check(o, lse, o_ref, l_ref)


def test_fwd_is_deterministic_and_overwrites_outputs():
    w = Workload("det", b=1, s=1024, hq=4, hkv=2, d=128, cp=2, seed=5)
    x = make_inputs(w, device="cuda")
    o1 = torch.full_like(x["q"], float("nan"))
    l1 = torch.full((1, 4, 1024), float("nan"), device="cuda")
    cpattn_fwd(x["q"], x["k"], x["v"], 2, o=o1, lse=l1)
    o2, l2 = cpattn_fwd(x["q"], x["k"], x["v"], 2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_cp_degree_does_not_change_result():
    """The CP split only reorders the key walk: any cp gives the same attention."""
    w = Workload("cpinv", b=1, s=3072, hq=2, hkv=1, d=128, cp=1, seed=9)
    x = make_inputs(w, device="cuda")
    outs = [cpattn_fwd(x["q"], x["k"], x["v"], cp) for cp in (1, 2, 3, 4, 6, 12)]
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2 * O_TOL
        assert (l - outs[0][1]).abs().max().item() <= 2 * LSE_TOL


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_fwd_full_size_workloads(name):
    w = WORKLOADS[name]
    x = make_inputs(w, device="cuda", with_grad=False)
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], w.cp, causal=w.causal)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    rows = None if w.check_rows == 0 else sample_rows(w, w.check_rows, seed=w.seed + 77)
    o_c, lse_c = o.cpu(), lse.cpu()
    del o, lse
    # the computation's own error, without the bf16 output rounding: fp32 O
    # through the CP steps must meet the bar with no allowance
    o32, l32 = _fp32_o_by_steps(x["q"], x["k"], x["v"], w.cp, w.causal)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    o32_c = (o32 if rows is None else o32[:, rows.to(o32.device)]).double().cpu()
    l32_c = (l32 if rows is None else l32[:, :, rows.to(l32.device)]).double().cpu()
    del o32, l32
    q_c, k_c, v_c = x["q"].cpu(), x["k"].cpu(), x["v"].cpu()
    del x
    o_ref, l_ref = oracle.attention_forward(q_c, k_c, v_c, causal=w.causal, rows=rows,
                                            row_block=128 if w.s > 32768 else 512)
    _check(o_c, lse_c, o_ref, l_ref, rows=rows, name=name)
    raw32 = (o32_c - o_ref).abs().max().item()
    l32_err = (l32_c - l_ref).abs().max().item()
    print(f"PARITY {name} fp32 O through the CP steps: max|O err| raw {raw32:.3e}, max|LSE err| {l32_err:.3e}")
    assert raw32 <= O_TOL and l32_err <= LSE_TOL


def test_fwd_tile_pair_blocks_match_unblocked_bitwise():
    """Odd head groups (G = 3, tile pairs) whose K/V outgrows L2 (b8 s4096 hq24
    hkv8: 128 MB) run their units in L2-sized head blocks; one batch element
    alone (16 MB) runs them unblocked. The units are the same, only their
    order differs, so every batch element's output is bit-identical to its
    own launch; sampled rows of two elements also meet the oracle bar."""
    w = Workload("tp_blocks", b=8, s=4096, hq=24, hkv=8, d=128, cp=4, seed=4242)
    x = make_inputs(w, device="cuda", with_grad=False)
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], w.cp)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    for bi in range(w.b):
        one = [x[n][bi:bi + 1].contiguous() for n in ("q", "k", "v")]
        o1, l1 = cpattn_fwd(*one, w.cp)
        torch.cuda.synchronize()
        assert torch.equal(o1[0], o[bi]) and torch.equal(l1[0], lse[bi]), f"batch element {bi}"
    rows = sample_rows(w, 48, seed=9)
    for bi in (0, w.b - 1):
        o_ref, l_ref = oracle.attention_forward(*[x[n][bi:bi + 1].cpu() for n in ("q", "k", "v")], rows=rows)
        _check(o[bi:bi + 1, rows].cpu(), lse[bi:bi + 1][:, :, rows].cpu(), o_ref, l_ref, name=f"tp_blocks b{bi}")


@pytest.mark.parametrize("d", [128, 64])
def test_fwd_output_only_16_byte_aligned(d):
    """The ABI asks o for 16-byte alignment only: an o 16 bytes past a 32-byte
    boundary gets the same result as an aligned one, bit for bit, and nothing
    around it is written."""
    w = Workload("off16", b=2, s=1024, hq=4, hkv=2, d=d, cp=2, seed=5)
    x = make_inputs(w, device="cuda", with_grad=False)
    o_ref, l_ref = cpattn_fwd(x["q"], x["k"], x["v"], w.cp)
    buf = torch.zeros(x["q"].numel() + 16, dtype=torch.bfloat16, device="cuda")
    o_off = buf[8:8 + x["q"].numel()].view(x["q"].shape)
    assert o_off.data_ptr() % 32 == 16
    o2, l2 = cpattn_fwd(x["q"], x["k"], x["v"], w.cp, o=o_off)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    assert torch.equal(o2, o_ref) and torch.equal(l2, l_ref)
    assert not buf[:8].any() and not buf[8 + x["q"].numel():].any()  # nothing outside o written


@pytest.mark.parametrize("std,cp,d", [(8.0, 4, 128), (16.0, 2, 64)])
def test_fwd_peaky_scores_all_elements(std, cp, d):
    """Q, K ~ N(0, std^2): scores of several hundred, a row's maximum moves
    often and most probabilities underflow; every element against the
    oracle."""
    w = Workload("peaky", b=1, s=1024, hq=4, hkv=2, d=d, cp=cp, q_std=std, k_std=std, seed=31 + cp)
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], cp)
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    o_ref, l_ref = oracle.attention_forward(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), causal=True)
    _check(o, lse, o_ref, l_ref)

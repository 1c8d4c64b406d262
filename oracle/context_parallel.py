"""The context-parallel procedure itself, emulated on the CPU in fp64.

TEST INFRASTRUCTURE (see the package docstring).

This is a second, independent route to the attention result: it follows the
steps the pages give for Megatron-LM's CP instead of the plain definition,
so agreement between the two pins both.

Split ([MLM-CP] 3.2 step 1 and 3.4; [Practice] "CP 与其他技术结合"): the
sequence of s tokens is cut into 2*cp chunks of c = s/(2cp) tokens; virtual
rank r holds chunk r and its mirror chunk 2cp-1-r (rank 0 trades half of its
data with rank cp-1, rank 1 with rank cp-2, ...), so every rank has one
"small" and one "large" causal workload.

Steps ([MLM-CP] 3.2 steps 2-5, 3.4): at step i the rank holds the KV of
source rank j = (r - i) mod cp (the ring of 3.2 step 3, one hop per step).
  * step 0: local Q (both chunks) against local KV (both chunks), causal;
  * 1 <= i <= r: all local Q against the first half of the incoming KV
    (chunk j), no mask;
  * i > r: only the second half of Q (chunk 2cp-1-r) against the full
    incoming KV (chunks j and 2cp-1-j), no mask.
Reading taken: "first half" of a rank's pair is its lower-position chunk;
it is the only reading under which these blocks need no mask. Each step
yields a partial output O_i and log-sum-exp L_i over its own keys; L is
corrected after every step and the O_i are corrected and merged at the end
(3.2 steps 4-5). The correction formulas were lost from the page (the FA2
figure of 3.3); they are taken as the standard two-stage log-sum-exp, the
same algebra as [M019]'s global max / global exp-sum:
    L = log(sum_i exp(L_i)),   O = sum_i exp(L_i - L) * O_i.

With causal=False every step is unmasked over all local Q and the full
incoming KV pair.
"""
import math

import torch

_F64 = torch.float64


def zigzag_chunks(cp: int):
    """[(r, (first_chunk, second_chunk))] for every virtual rank r."""
    if cp < 1:
        raise ValueError("cp must be >= 1")
    return [(r, (r, 2 * cp - 1 - r)) for r in range(cp)]


def zigzag_global_index(s: int, cp: int) -> torch.Tensor:
    """int64 [cp, 2c]: global token position of rank r's local position u.

    Local order is [chunk r, chunk 2cp-1-r], each in natural order.
    """
    if s % (2 * cp) != 0:
        raise ValueError("s must be divisible by 2*cp")
    c = s // (2 * cp)
    out = torch.empty(cp, 2 * c, dtype=torch.long)
    for r, (lo, hi) in zigzag_chunks(cp):
        for u in range(2 * c):
            out[r, u] = lo * c + u if u < c else hi * c + (u - c)
    return out


def cp_step_plan(r: int, cp: int, causal: bool = True):
    """The blocks rank r computes, step by step.

    Returns a list of (step, source_rank, q_chunks, kv_chunks, masked):
    chunk ids are global chunk indices; ``masked`` means the step applies the
    causal mask (step 0 only).
    """
    lo, hi = r, 2 * cp - 1 - r
    plan = []
    for i in range(cp):
        j = (r - i) % cp
        j_lo, j_hi = j, 2 * cp - 1 - j
        if not causal:
            plan.append((i, j, (lo, hi), (j_lo, j_hi), False))
        elif i == 0:
            plan.append((i, j, (lo, hi), (lo, hi), True))
        elif i <= r:
            plan.append((i, j, (lo, hi), (j_lo,), False))
        else:
            plan.append((i, j, (hi,), (j_lo, j_hi), False))
    return plan


def block_attention(qb, kb, vb, q_pos, k_pos, masked, scale):
    """One step's block: softmax over this block's keys only.

    qb [n, d], kb/vb [m, d]; q_pos/k_pos global positions (used for the mask).
    Returns (O_i [n, d], L_i [n]); rows that see no key in the block get
    L_i = -inf and O_i = 0 (they drop out of the merge).
    """
    S = (qb @ kb.T) * scale
    if masked:
        S = S.masked_fill(k_pos[None, :] > q_pos[:, None], float("-inf"))
    m = S.max(dim=1, keepdim=True).values
    m_safe = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
    e = torch.exp(S - m_safe)
    l = e.sum(dim=1, keepdim=True)
    L = torch.where(l > 0, m_safe + torch.log(l), torch.full_like(l, float("-inf")))
    O = torch.where(l > 0, e / torch.where(l > 0, l, torch.ones_like(l)), torch.zeros_like(e)) @ vb
    return O, L[:, 0]


def lse_merge(parts):
    """Merge partial results [(O_i [n, d], L_i [n]), ...] over disjoint key sets.

    Stage 1 corrects L after every part (running log-add-exp); stage 2
    corrects each O_i by exp(L_i - L) and sums them.
    """
    if not parts:
        raise ValueError("nothing to merge")
    L = parts[0][1].clone()
    for _, Li in parts[1:]:
        m = torch.maximum(L, Li)
        m_safe = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
        L = torch.where(torch.isfinite(m), m_safe + torch.log(torch.exp(L - m_safe) + torch.exp(Li - m_safe)), m)
    O = torch.zeros_like(parts[0][0])
    for Oi, Li in parts:
        w = torch.where(torch.isfinite(L), torch.exp(Li - torch.where(torch.isfinite(L), L, torch.zeros_like(L))),
                        torch.zeros_like(L))
        O = O + w[:, None] * Oi
    return O, L


def cp_step_partials(q, k, v, cp, step, causal=True):
    """Every virtual rank's partial result of one CP step, in natural order.

    q: [b, s, hq, d]; k, v: [b, s, hkv, d]; float64 CPU. At step ``step``
    rank r computes the block of ``cp_step_plan(r, cp, causal)[step]``
    ([MLM-CP] 3.2 steps 2-3, 3.4). Returns (o_i [b, s, hq, d], lse_i
    [b, hq, s]): for the query rows of those blocks the block's own softmax
    output and log-sum-exp (before any correction, 3.2 step 4); every other
    row gets O = 0 and L = -inf, so merging all steps' partials with
    ``lse_merge`` row by row gives the attention result.
    """
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    G = hq // hkv
    c = s // (2 * cp)
    scale = 1.0 / math.sqrt(d)
    o = torch.zeros(b, s, hq, d, dtype=_F64)
    lse = torch.full((b, hq, s), float("-inf"), dtype=_F64)

    def chunk_pos(ch):
        return torch.arange(ch * c, (ch + 1) * c, dtype=torch.long)

    for bi in range(b):
        for h in range(hq):
            g = h // G
            for r in range(cp):
                _i, _j, q_ch, kv_ch, masked = cp_step_plan(r, cp, causal)[step]
                q_pos = torch.cat([chunk_pos(ch) for ch in q_ch])
                k_pos = torch.cat([chunk_pos(ch) for ch in kv_ch])
                Oi, Li = block_attention(q[bi, q_pos, h], k[bi, k_pos, g], v[bi, k_pos, g], q_pos, k_pos, masked,
                                         scale)
                o[bi, q_pos, h] = Oi
                lse[bi, h, q_pos] = Li
    return o, lse


def cp_attention_forward(q, k, v, cp, causal=True, merge_order=None):
    """Attention computed the CP way: per virtual rank, per step, then merged.

    q: [b, s, hq, d]; k, v: [b, s, hkv, d]; float64 CPU. Returns (o, lse) in
    natural token order, shaped like ``attention_forward``'s. ``merge_order``
    (optional callable: list of step indices -> permuted list) changes the
    order in which a rank merges its partial results.
    """
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    G = hq // hkv
    c = s // (2 * cp)
    scale = 1.0 / math.sqrt(d)
    gidx = zigzag_global_index(s, cp)
    o = torch.zeros(b, s, hq, d, dtype=_F64)
    lse = torch.full((b, hq, s), float("-inf"), dtype=_F64)

    def chunk_pos(ch):
        return torch.arange(ch * c, (ch + 1) * c, dtype=torch.long)

    for bi in range(b):
        for h in range(hq):
            g = h // G
            for r in range(cp):
                local = gidx[r]  # global position of each local row
                parts_per_row = [[] for _ in range(2 * c)]
                for (_i, _j, q_ch, kv_ch, masked) in cp_step_plan(r, cp, causal):
                    q_pos = torch.cat([chunk_pos(ch) for ch in q_ch])
                    k_pos = torch.cat([chunk_pos(ch) for ch in kv_ch])
                    Oi, Li = block_attention(q[bi, q_pos, h], k[bi, k_pos, g], v[bi, k_pos, g], q_pos, k_pos,
                                             masked, scale)
                    for n, t in enumerate(q_pos.tolist()):
                        u = t - r * c if t < (r + 1) * c else c + (t - (2 * cp - 1 - r) * c)
                        parts_per_row[u].append((Oi[n:n + 1], Li[n:n + 1]))
                for u in range(2 * c):
                    parts = parts_per_row[u]
                    if merge_order is not None:
                        parts = [parts[idx] for idx in merge_order(list(range(len(parts))))]
                    Ou, Lu = lse_merge(parts)
                    t = int(local[u])
                    o[bi, t, h] = Ou[0]
                    lse[bi, h, t] = Lu[0]
    return o, lse

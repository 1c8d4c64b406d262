"""Uncut causal softmax attention and its gradients, fp64 on the CPU.

TEST INFRASTRUCTURE (see the package docstring): imported only by tests, the
smoke check and the bench's CPU-baseline leg.

Definition followed ([MLM-CP] 3.2: every rank's output equals the matching
rows of the result computed without CP, so the oracle is that uncut result).
For batch b, query head h with KV head g = h // G (G = hq / hkv, [M014] and
[Practice] on GQA: a group of query heads shares one K and one V), query t:

    S[t, j] = scale * <q[b,t,h], k[b,j,g]>        for j <= t (all j if not causal)
    L[t]    = log sum_j exp(S[t, j])               (natural log)
    O[t]    = sum_j exp(S[t, j] - L[t]) * v[b,j,g]

scale = 1/sqrt(d). Rows are independent by this definition, so they are
processed in blocks only to bound memory; keys past the last row of a block
are masked for every row in it and are not formed. Library steps used: a
matmul, exp, log, max and sum (torch, float64, CPU).
"""
import math

import torch

_F64 = torch.float64


def softmax_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


_EXACT = (torch.bfloat16, torch.float16, torch.float32, torch.float64)


def _check(q, k, v):
    # Inputs may be bf16/fp16/fp32/fp64: each block is upcast to float64,
    # which is exact for all of them; all arithmetic is float64.
    if q.dtype not in _EXACT or k.dtype not in _EXACT or v.dtype not in _EXACT:
        raise TypeError("oracle inputs must be a float type that upcasts exactly to float64")
    if q.device.type != "cpu":
        raise ValueError("oracle runs on the CPU")
    b, s, hq, d = q.shape
    if k.shape[0] != b or k.shape[3] != d or v.shape != k.shape or hq % k.shape[2] != 0:
        raise ValueError("shape mismatch")
    return b, s, hq, d, k.shape[1], k.shape[2]


def _rows_tensor(rows, s):
    if rows is None:
        return torch.arange(s, dtype=torch.long)
    return torch.as_tensor(rows, dtype=torch.long).reshape(-1)


def _scores(qrows, kk, t, causal, scale):
    """S = scale * q k^T over keys [0, kk.shape[0]), masked to j <= t."""
    S = (qrows @ kk.T) * scale
    if causal:
        j = torch.arange(kk.shape[0], dtype=torch.long)
        S.masked_fill_(j[None, :] > t[:, None], float("-inf"))
    return S


def attention_forward(q, k, v, causal=True, rows=None, row_block=1024, scale=None):
    """O and LSE of softmax attention for the query positions ``rows``.

    Scores are ``scale * q.k`` (default scale 1/sqrt(d)).

    q: [b, s, hq, d]; k, v: [b, s_kv, hkv, d]; CPU tensors of a float type
    that upcasts exactly (bf16, fp16, fp32, fp64); arithmetic is float64.
    Returns o [b, n, hq, d] and lse [b, hq, n] (n = len(rows), default all s).
    A row that sees no key (impossible for causal self-attention) gets
    L = -inf and O = 0.
    """
    b, s, hq, d, skv, hkv = _check(q, k, v)
    G = hq // hkv
    scale = softmax_scale(d) if scale is None else float(scale)
    t_all = _rows_tensor(rows, s)
    n = t_all.numel()
    o = torch.zeros(b, n, hq, d, dtype=_F64)
    lse = torch.empty(b, hq, n, dtype=_F64)
    for bi in range(b):
        for g in range(hkv):
            kk_all = k[bi, :, g].to(_F64)
            vv_all = v[bi, :, g].to(_F64)
            for h in range(g * G, (g + 1) * G):
                for r0 in range(0, n, row_block):
                    t = t_all[r0:r0 + row_block]
                    nk = min(int(t.max()) + 1, skv) if causal else skv
                    S = _scores(q[bi, t, h].to(_F64), kk_all[:nk], t, causal, scale)
                    m = S.max(dim=1, keepdim=True).values
                    m_safe = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
                    L = m_safe + torch.log(torch.exp(S - m_safe).sum(dim=1, keepdim=True))
                    P = torch.exp(S - torch.where(torch.isfinite(L), L, torch.zeros_like(L)))
                    P = torch.where(torch.isfinite(L), P, torch.zeros_like(P))
                    o[bi, r0:r0 + t.numel(), h] = P @ vv_all[:nk]
                    lse[bi, h, r0:r0 + t.numel()] = L[:, 0]
    return o, lse


def attention_backward(q, k, v, do, causal=True, dq_rows=None, dkv_heads=None, row_block=512, scale=None):
    """Gradients of sum(dO * O) with respect to q, k and v.

    With P = softmax(S) row-wise and O = P V (the forward above):
        dV[j] = sum_t P[t, j] dO[t]
        dP[t, j] = <dO[t], v[j]>
        dS[t, j] = P[t, j] * (dP[t, j] - sum_i P[t, i] dP[t, i])   (softmax Jacobian)
        dQ[t] = scale * sum_j dS[t, j] k[j]
        dK[j] = scale * sum_t dS[t, j] q[t]
    dK and dV of KV head g sum over every query head of g's group.

    ``scale``: the forward's score scale (default 1/sqrt(d)).
    ``dq_rows``: query positions whose dQ is wanted (default: all).
    ``dkv_heads``: KV heads whose dK/dV are wanted (default: all); these need
    every row of every query head in the group.
    Returns (dq [b, n_rows, hq, d], dk [b, s_kv, n_heads, d], dv likewise);
    dk/dv carry only the requested heads, in the order given.
    """
    b, s, hq, d, skv, hkv = _check(q, k, v)
    if do.shape != q.shape or do.dtype not in _EXACT:
        raise ValueError("do must match q")
    G = hq // hkv
    scale = softmax_scale(d) if scale is None else float(scale)
    t_dq = _rows_tensor(dq_rows, s)
    heads = list(range(hkv)) if dkv_heads is None else [int(g) for g in dkv_heads]
    dq = torch.zeros(b, t_dq.numel(), hq, d, dtype=_F64)
    dk = torch.zeros(b, skv, len(heads), d, dtype=_F64)
    dv = torch.zeros(b, skv, len(heads), d, dtype=_F64)

    def grads_for_rows(qq, kk, vv, dd, t):
        nk = min(int(t.max()) + 1, skv) if causal else skv
        S = _scores(qq, kk[:nk], t, causal, scale)
        m = S.max(dim=1, keepdim=True).values
        P = torch.exp(S - m)
        P = P / P.sum(dim=1, keepdim=True)
        dP = dd @ vv[:nk].T
        dS = P * (dP - (P * dP).sum(dim=1, keepdim=True))
        return nk, P, dS

    for bi in range(b):
        for g in range(hkv):
            kk = k[bi, :, g].to(_F64)
            vv = v[bi, :, g].to(_F64)
            for h in range(g * G, (g + 1) * G):
                # dQ on the requested rows
                for r0 in range(0, t_dq.numel(), row_block):
                    t = t_dq[r0:r0 + row_block]
                    nk, P, dS = grads_for_rows(q[bi, t, h].to(_F64), kk, vv, do[bi, t, h].to(_F64), t)
                    dq[bi, r0:r0 + t.numel(), h] = scale * (dS @ kk[:nk])
                # dK / dV of the requested KV heads: every row of this query head
                if g in heads:
                    slot = heads.index(g)
                    t_all = torch.arange(s, dtype=torch.long)
                    for r0 in range(0, s, row_block):
                        t = t_all[r0:r0 + row_block]
                        qq = q[bi, t, h].to(_F64)
                        dd = do[bi, t, h].to(_F64)
                        nk, P, dS = grads_for_rows(qq, kk, vv, dd, t)
                        dv[bi, :nk, slot] += P.T @ dd
                        dk[bi, :nk, slot] += scale * (dS.T @ qq)
    return dq, dk, dv

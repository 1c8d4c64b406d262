"""Attention over packed samples, fp64 on the CPU. TEST INFRASTRUCTURE (see
the package docstring).

Packing ("Megatron 面试题（一）：模型抽象与训练数据流", item M016, follow-up:
sample boundaries under CP) puts several samples back to back in one
sequence; attention must not cross a sample boundary. Each sample is thus
its own attention problem (under CP each sample is split by the zigzag on
its own; the result is the sample's plain attention either way, by the
equality of the CP route and the uncut one).
"""
import torch

from .attention import attention_backward, attention_forward

_F64 = torch.float64


def _slices(cu):
    cu = [int(x) for x in cu]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def varlen_attention_forward(q, k, v, cu_seqlens, causal=True, scale=None):
    """q [total, hq, d], k/v [total, hkv, d]: (o [total, hq, d], lse [hq, total])."""
    total, hq, d = q.shape
    o = torch.zeros(total, hq, d, dtype=_F64)
    lse = torch.full((hq, total), float("-inf"), dtype=_F64)
    for a, b in _slices(cu_seqlens):
        if b == a:
            continue
        oi, li = attention_forward(q[None, a:b], k[None, a:b], v[None, a:b], causal=causal, scale=scale)
        o[a:b] = oi[0]
        lse[:, a:b] = li[0]
    return o, lse


def varlen_attention_backward(q, k, v, do, cu_seqlens, causal=True, scale=None):
    """Gradients of sum(dO * O) over packed samples: (dq, dk, dv) shaped like q, k, v."""
    dq = torch.zeros(q.shape, dtype=_F64)
    dk = torch.zeros(k.shape, dtype=_F64)
    dv = torch.zeros(v.shape, dtype=_F64)
    for a, b in _slices(cu_seqlens):
        if b == a:
            continue
        gq, gk, gv = attention_backward(q[None, a:b], k[None, a:b], v[None, a:b], do[None, a:b], causal=causal,
                                        scale=scale)
        dq[a:b], dk[a:b], dv[a:b] = gq[0], gk[0], gv[0]
    return dq, dk, dv

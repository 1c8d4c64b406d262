"""Rotary position embedding (RoPE) with the positions context parallelism
needs, fp64 on the CPU. TEST INFRASTRUCTURE (see the package docstring).

RoPE rotates query and key vectors inside attention by an angle that grows
with the token's position, so that q_m . k_n depends on m - n only ("Megatron
面试题（一）：模型抽象与训练数据流", item M016: RoPE acts on Q/K inside
attention and adds no position table). Under CP a rank holds only its two
zigzag chunks, yet the phase must be that of the token's position in the
whole sequence -- renumbering local tokens from 0 would break the relative
phases across chunks -- and with packed samples the position restarts at
each sample boundary (same item, follow-up answer).

Form used (the pages give none; this is the common "half rotation" layout):
for head dimension d, each pair (x_i, x_{i+d/2}), i < d/2, is rotated by
theta = pos * base^(-2i/d):
    x_i'       = x_i cos(theta) - x_{i+d/2} sin(theta)
    x_{i+d/2}' = x_i sin(theta) + x_{i+d/2} cos(theta).
"""
import torch

from .context_parallel import zigzag_global_index

_F64 = torch.float64


def rope_angles(pos, d, base=10000.0):
    """theta[n, d/2] for integer positions ``pos`` [n]."""
    i = torch.arange(d // 2, dtype=_F64)
    inv_freq = base ** (-2.0 * i / d)
    return pos.to(_F64)[:, None] * inv_freq[None, :]


def rope_apply(x, pos, base=10000.0, inverse=False):
    """Rotate x [b, n, h, d] (float64) at positions pos [n] (or [b, n])."""
    b, n, h, d = x.shape
    half = d // 2
    pos = pos if pos.dim() == 2 else pos[None, :].expand(b, n)
    out = torch.empty_like(x, dtype=_F64)
    for bi in range(b):
        th = rope_angles(pos[bi], d, base)  # [n, d/2]
        c, s = torch.cos(th)[:, None, :], torch.sin(th)[:, None, :]
        if inverse:
            s = -s
        x1, x2 = x[bi, :, :, :half].to(_F64), x[bi, :, :, half:].to(_F64)
        out[bi, :, :, :half] = x1 * c - x2 * s
        out[bi, :, :, half:] = x1 * s + x2 * c
    return out


def natural_positions(s, cu_seqlens=None):
    """Position of each token of a natural-order sequence of s tokens: its
    index, or with packing (``cu_seqlens`` = sample start offsets, ending
    with s) its index within its sample."""
    t = torch.arange(s, dtype=torch.long)
    if cu_seqlens is None:
        return t
    cu = torch.as_tensor(cu_seqlens, dtype=torch.long)
    start = cu[torch.searchsorted(cu, t, right=True) - 1]
    return t - start


def rank_local_positions(s, cp, r, cu_seqlens=None):
    """Positions of virtual rank r's 2c local tokens (chunk r, then chunk
    2cp-1-r): the global positions of the zigzag map, not 0..2c-1."""
    g = zigzag_global_index(s, cp)[r]
    return natural_positions(s, cu_seqlens)[g]

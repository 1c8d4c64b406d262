"""GB300-native context-parallel causal attention.

Python binding of the C-ABI library ``libcpattn.so`` (include/cpattn.h).
This module only marshals arguments: it checks tensor properties, allocates
outputs with PyTorch when the caller does not pass them, and hands raw device
pointers, sizes and the current CUDA stream to the library. Every step of the
computation runs in the library's CUDA kernels; there is no fallback. If the
library has not been built the calls raise.
"""
import ctypes
import os

import torch

from ._build import CHECKED_LIB_PATH, LIB_PATH, build  # noqa: F401

__all__ = [
    "CpattnError",
    "cpattn_set_max_ctas",
    "cpattn_fwd",
    "cpattn_fwd_step",
    "cpattn_lse_merge",
    "cpattn_fwd_unfused",
    "cpattn_fwd_unfused_workspace_bytes",
    "cpattn_rope",
    "cpattn_fwd_varlen",
    "cpattn_bwd_varlen",
    "cpattn_bwd",
    "cpattn_bwd_workspace_bytes",
    "cpattn_zigzag_index",
    "cpattn_fwd_rank",
    "cpattn_fwd_rank_step",
    "cpattn_bwd_rank",
    "cpattn_bwd_rank_workspace_bytes",
    "cpattn_device_status",
    "cpattn_selftest_wait_timeout",
    "library",
]

CPATTN_ERRORS = {
    -1: "CPATTN_ERR_INVALID_ARG",
    -2: "CPATTN_ERR_NULL_PTR",
    -3: "CPATTN_ERR_MISALIGNED",
    -4: "CPATTN_ERR_UNSUPPORTED_ARCH",
    -5: "CPATTN_ERR_WORKSPACE_TOO_SMALL",
    -6: "CPATTN_ERR_LAUNCH_FAILED",
    -7: "CPATTN_ERR_TIMEOUT",
    -8: "CPATTN_ERR_CUDA",
}


class CpattnError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        lib = _LIB
        msg = lib.cpattn_strerror(code).decode() if lib is not None else CPATTN_ERRORS.get(code, "error")
        super().__init__(f"{what}: {CPATTN_ERRORS.get(code, code)} ({msg})")


_LIB = None
_i, _p, _sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t


_CHECKED = None


def library():
    """Load libcpattn.so (once). Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with context_blockwise_causal_gb300.build()")
        _LIB = _declare(ctypes.CDLL(LIB_PATH))
    return _LIB


def checked_library():
    """Load libcpattn_checked.so (once), the build whose kernels test every
    global access against the buffers' extents (bit 20 of the status word).
    A debugging aid with the same entry points and results; raises if it has
    not been built."""
    global _CHECKED
    if _CHECKED is None:
        if not os.path.exists(CHECKED_LIB_PATH):
            raise RuntimeError(f"{CHECKED_LIB_PATH} is missing: build it with context_blockwise_causal_gb300.build()")
        _CHECKED = _declare(ctypes.CDLL(CHECKED_LIB_PATH))
    return _CHECKED


def _declare(lib):
    """Argument and result types of every entry point of a loaded library."""
    lib.cpattn_set_max_ctas.argtypes = [_i]
    lib.cpattn_set_max_ctas.restype = _i
    lib.cpattn_fwd.argtypes = [_p, _p, _p, _p, _p] + [_i] * 7 + [_p]
    lib.cpattn_fwd.restype = _i
    lib.cpattn_fwd_ex.argtypes = [_p, _p, _p, _p, _p] + [_i] * 7 + [ctypes.c_float, _p]
    lib.cpattn_fwd_ex.restype = _i
    lib.cpattn_bwd_ex.argtypes = [_p] * 10 + [_sz] + [_i] * 7 + [ctypes.c_float, _p]
    lib.cpattn_bwd_ex.restype = _i
    lib.cpattn_fwd_step.argtypes = [_p] * 5 + [_i] * 8 + [_p]
    lib.cpattn_fwd_step.restype = _i
    lib.cpattn_lse_merge.argtypes = [_p] * 7 + [_i] * 4 + [_p]
    lib.cpattn_lse_merge.restype = _i
    lib.cpattn_fwd_unfused_workspace_bytes.argtypes = [_i] * 4
    lib.cpattn_fwd_unfused_workspace_bytes.restype = _sz
    lib.cpattn_fwd_unfused.argtypes = [_p] * 6 + [_sz] + [_i] * 7 + [_p]
    lib.cpattn_fwd_unfused.restype = _i
    lib.cpattn_rope.argtypes = [_p] + [_i] * 7 + [_p, _i, ctypes.c_float, _i, _p]
    lib.cpattn_rope.restype = _i
    lib.cpattn_fwd_varlen.argtypes = [_p] * 6 + [_i] * 6 + [ctypes.c_float, _p]
    lib.cpattn_fwd_varlen.restype = _i
    lib.cpattn_bwd_varlen_workspace_bytes.argtypes = [_p] + [_i] * 5
    lib.cpattn_bwd_varlen_workspace_bytes.restype = _sz
    lib.cpattn_bwd_varlen.argtypes = [_p] * 10 + [_sz, _p] + [_i] * 6 + [ctypes.c_float, _p]
    lib.cpattn_bwd_varlen.restype = _i
    lib.cpattn_bwd.argtypes = [_p] * 10 + [_sz] + [_i] * 7 + [_p]
    lib.cpattn_bwd.restype = _i
    lib.cpattn_bwd_stage.argtypes = [_i] + [_p] * 10 + [_sz] + [_i] * 7 + [_p]
    lib.cpattn_bwd_stage.restype = _i
    lib.cpattn_bwd_noalloc.argtypes = [_p] * 9 + [_i] * 7 + [_p]
    lib.cpattn_bwd_noalloc.restype = _i
    lib.cpattn_bwd_noalloc_max_scratch_bytes.argtypes = []
    lib.cpattn_bwd_noalloc_max_scratch_bytes.restype = _sz
    lib.cpattn_bwd_workspace_bytes.argtypes = [_i] * 6
    lib.cpattn_bwd_workspace_bytes.restype = _sz
    lib.cpattn_fwd_rank.argtypes = [_p] * 5 + [_i] * 8 + [ctypes.c_float, _p]
    lib.cpattn_fwd_rank.restype = _i
    lib.cpattn_fwd_rank_step.argtypes = [_p] * 5 + [_i] * 9 + [ctypes.c_float, _p]
    lib.cpattn_fwd_rank_step.restype = _i
    lib.cpattn_bwd_rank_workspace_bytes.argtypes = [_i] * 6
    lib.cpattn_bwd_rank_workspace_bytes.restype = _sz
    lib.cpattn_bwd_rank.argtypes = [_p] * 10 + [_sz] + [_i] * 8 + [ctypes.c_float, _p]
    lib.cpattn_bwd_rank.restype = _i
    lib.cpattn_bwd_rank_stage.argtypes = [_i] + [_p] * 10 + [_sz] + [_i] * 8 + [ctypes.c_float, _p]
    lib.cpattn_bwd_rank_stage.restype = _i
    lib.cpattn_zigzag_index.argtypes = [_i, _i, _p]
    lib.cpattn_zigzag_index.restype = _i
    lib.cpattn_device_status.argtypes = [_p, ctypes.POINTER(_i)]
    lib.cpattn_device_status.restype = _i
    lib.cpattn_selftest_abort.argtypes = [_p] * 10 + [_sz] + [_i] * 6 + [ctypes.c_ulonglong, _p]
    lib.cpattn_selftest_abort.restype = _i
    lib.cpattn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, _p]
    lib.cpattn_selftest_wait_timeout.restype = _i
    lib.cpattn_strerror.argtypes = [_i]
    lib.cpattn_strerror.restype = ctypes.c_char_p
    lib.cpattn_version.argtypes = []
    lib.cpattn_version.restype = _i
    lib.cpattn_checked_build.argtypes = []
    lib.cpattn_checked_build.restype = _i
    lib.cpattn_selftest_bounds.argtypes = [_p] * 5 + [_i] * 6 + [_p]
    lib.cpattn_selftest_bounds.restype = _i
    return lib


def _stream_handle(stream, *tensors):
    """The stream to launch on (the current one by default). The library
    launches on the current CUDA device, so every tensor given must be on it,
    and so must the stream."""
    cur = torch.cuda.current_device()
    for t in tensors:
        if isinstance(t, torch.Tensor) and t.is_cuda and t.device.index != cur:
            raise ValueError(f"a tensor is on {t.device} but the current CUDA device is cuda:{cur}; "
                             f"call under torch.cuda.device({t.device})")
    if stream is None:
        stream = torch.cuda.current_stream()
    elif stream.device.index != cur:
        raise ValueError(f"the stream belongs to {stream.device}, the current CUDA device is cuda:{cur}")
    return ctypes.c_void_p(stream.cuda_stream)


def _check_act(name, t, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dims(q, k, v):
    _check_act("q", q)
    if q.dim() != 4:
        raise ValueError("q must be [b, s, hq, d]")
    b, s, hq, d = q.shape
    _check_act("k", k)
    if k.dim() != 4 or k.shape[0] != b or k.shape[1] != s or k.shape[3] != d:
        raise ValueError("k must be [b, s, hkv, d]")
    _check_act("v", v, k.shape)
    return b, s, hq, k.shape[2], d


def cpattn_fwd(q, k, v, cp, causal=True, o=None, lse=None, stream=None, scale=None):
    """Context-parallel causal attention forward. Returns (o, lse).

    q [b,s,hq,d], k/v [b,s,hkv,d] bf16 CUDA tensors; o like q (bf16) and lse
    [b,hq,s] fp32 are allocated when not given. ``scale`` (default 1/sqrt(d))
    multiplies the scores (cpattn_fwd_ex).
    """
    b, s, hq, hkv, d = _dims(q, k, v)
    if o is None:
        o = torch.empty_like(q)
    _check_act("o", o, q.shape)
    if lse is None:
        lse = torch.empty(b, hq, s, device=q.device, dtype=torch.float32)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (b, hq, s) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [b, hq, s] tensor")
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), b, s, hq, hkv, d, int(cp),
            1 if causal else 0)
    if scale is None:
        rc = library().cpattn_fwd(*args, _stream_handle(stream, q, k, v, o, lse))
    else:
        rc = library().cpattn_fwd_ex(*args, float(scale), _stream_handle(stream, q, k, v, o, lse))
    if rc:
        raise CpattnError(rc, "cpattn_fwd" if scale is None else "cpattn_fwd_ex")
    return o, lse


def _check_f32(name, t, shape):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous fp32 CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def cpattn_fwd_step(q, k, v, cp, step, causal=True, o_part=None, lse_part=None, stream=None):
    """Every virtual rank's unmerged result of CP step ``step``.

    Returns (o_part [b,s,hq,d] fp32, lse_part [b,hq,s] fp32); rows that take
    no part in the step get 0 and -inf.
    """
    b, s, hq, hkv, d = _dims(q, k, v)
    if o_part is None:
        o_part = torch.empty(b, s, hq, d, device=q.device, dtype=torch.float32)
    if lse_part is None:
        lse_part = torch.empty(b, hq, s, device=q.device, dtype=torch.float32)
    _check_f32("o_part", o_part, (b, s, hq, d))
    _check_f32("lse_part", lse_part, (b, hq, s))
    rc = library().cpattn_fwd_step(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_part.data_ptr(), lse_part.data_ptr(),
                                   b, s, hq, hkv, d, int(cp), int(step), 1 if causal else 0,
                                   _stream_handle(stream, q, k, v, o_part, lse_part))
    if rc:
        raise CpattnError(rc, "cpattn_fwd_step")
    return o_part, lse_part


def cpattn_lse_merge(o_a, lse_a, o_b=None, lse_b=None, o_out=None, lse_out=None, o_bf16=None, stream=None):
    """Log-sum-exp merge of two partial results (fp32 [b,s,hq,d] / [b,hq,s]).

    Returns (o_out, lse_out, o_bf16); o_out may be ``o_a`` and lse_out
    ``lse_a`` (in place). With ``o_out=False`` no fp32 output is written
    (then ``o_bf16`` must be given or is allocated).
    """
    if o_a.dim() != 4:
        raise ValueError("o_a must be [b, s, hq, d]")
    b, s, hq, d = o_a.shape
    _check_f32("o_a", o_a, (b, s, hq, d))
    _check_f32("lse_a", lse_a, (b, hq, s))
    if (o_b is None) != (lse_b is None):
        raise ValueError("o_b and lse_b go together")
    if o_b is not None:
        _check_f32("o_b", o_b, (b, s, hq, d))
        _check_f32("lse_b", lse_b, (b, hq, s))
    if o_out is None:
        o_out = torch.empty_like(o_a)
    if o_out is not False:
        _check_f32("o_out", o_out, (b, s, hq, d))
    elif o_bf16 is None:
        o_bf16 = torch.empty(b, s, hq, d, device=o_a.device, dtype=torch.bfloat16)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    _check_f32("lse_out", lse_out, (b, hq, s))
    if o_bf16 is not None:
        _check_act("o_bf16", o_bf16, (b, s, hq, d))
    ptr = lambda t: None if t is None or t is False else t.data_ptr()  # noqa: E731
    rc = library().cpattn_lse_merge(ptr(o_a), ptr(lse_a), ptr(o_b), ptr(lse_b), ptr(o_out), ptr(lse_out),
                                    ptr(o_bf16), b, s, hq, d,
                                    _stream_handle(stream, o_a, lse_a, o_b, lse_b, o_out, lse_out, o_bf16))
    if rc:
        raise CpattnError(rc, "cpattn_lse_merge")
    return (None if o_out is False else o_out), lse_out, o_bf16


def cpattn_fwd_unfused_workspace_bytes(b, s, hq, d):
    return int(library().cpattn_fwd_unfused_workspace_bytes(b, s, hq, d))


def cpattn_fwd_unfused(q, k, v, cp, causal=True, o=None, lse=None, workspace=None, stream=None):
    """The forward as cp step launches and log-sum-exp merges. Returns (o, lse)."""
    b, s, hq, hkv, d = _dims(q, k, v)
    if o is None:
        o = torch.empty_like(q)
    _check_act("o", o, q.shape)
    if lse is None:
        lse = torch.empty(b, hq, s, device=q.device, dtype=torch.float32)
    _check_f32("lse", lse, (b, hq, s))
    need = cpattn_fwd_unfused_workspace_bytes(b, s, hq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    rc = library().cpattn_fwd_unfused(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      workspace.data_ptr(), workspace.numel() * workspace.element_size(), b, s, hq,
                                      hkv, d, int(cp), 1 if causal else 0,
                                      _stream_handle(stream, q, k, v, o, lse, workspace))
    if rc:
        raise CpattnError(rc, "cpattn_fwd_unfused")
    return o, lse


def cpattn_rope(x, base=10000.0, cp=1, rank=None, s=None, cu_seqlens=None, inverse=False, stream=None):
    """Rotary position embedding of x [b, n, h, d] bf16, in place; returns x.

    rank None: natural order (position = token index). rank r: x is virtual
    rank r's zigzag shard of a sequence of s tokens (n = s / cp).
    cu_seqlens: optional int32 CUDA tensor of packed-sample offsets (b == 1).
    """
    _check_act("x", x)
    if x.dim() != 4:
        raise ValueError("x must be [b, n, h, d]")
    b, n, h, d = x.shape
    if s is None:
        s = n if rank is None else n * cp
    cu_ptr, nseq = None, 0
    if cu_seqlens is not None:
        if not cu_seqlens.is_cuda or cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_contiguous():
            raise TypeError("cu_seqlens must be a contiguous int32 CUDA tensor")
        cu_ptr, nseq = cu_seqlens.data_ptr(), cu_seqlens.numel() - 1
    rc = library().cpattn_rope(x.data_ptr(), b, n, h, d, int(s), int(cp), -1 if rank is None else int(rank), cu_ptr,
                               nseq, float(base), 1 if inverse else 0, _stream_handle(stream, x, cu_seqlens))
    if rc:
        raise CpattnError(rc, "cpattn_rope")
    return x


def _cu_host(cu_seqlens):
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu().contiguous()
    return cu, ctypes.c_void_p(cu.data_ptr()), cu.numel() - 1


def _packed_dims(q, k, v):
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("packed q must be [total, hq, d] and k, v [total, hkv, d]")
    _check_act("q", q)
    _check_act("k", k)
    _check_act("v", v, k.shape)
    if k.shape[0] != q.shape[0] or k.shape[2] != q.shape[2]:
        raise ValueError("q and k disagree")
    return q.shape[0], q.shape[1], k.shape[1], q.shape[2]


def cpattn_fwd_varlen(q, k, v, cu_seqlens, cp, causal=True, scale=None, o=None, lse=None, stream=None):
    """Forward over packed samples (attention within each sample).

    q [total, hq, d], k/v [total, hkv, d]; cu_seqlens: sample offsets (host
    list/tensor). Returns (o [total, hq, d], lse [hq, total]).
    """
    total, hq, hkv, d = _packed_dims(q, k, v)
    cu, cu_p, nseq = _cu_host(cu_seqlens)
    if int(cu[-1]) != total:
        raise ValueError("cu_seqlens must end at the packed length")
    o = torch.empty_like(q) if o is None else o
    _check_act("o", o, q.shape)
    lse = torch.empty(hq, total, device=q.device, dtype=torch.float32) if lse is None else lse
    _check_f32("lse", lse, (hq, total))
    rc = library().cpattn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), cu_p,
                                     nseq, hq, hkv, d, int(cp), 1 if causal else 0,
                                     0.0 if scale is None else float(scale), _stream_handle(stream, q, k, v, o, lse))
    if rc:
        raise CpattnError(rc, "cpattn_fwd_varlen")
    return o, lse


def cpattn_bwd_varlen(q, k, v, o, lse, do, cu_seqlens, cp, causal=True, scale=None, dq=None, dk=None, dv=None,
                      workspace=None, stream=None):
    """Backward over packed samples. Returns (dq, dk, dv)."""
    total, hq, hkv, d = _packed_dims(q, k, v)
    cu, cu_p, nseq = _cu_host(cu_seqlens)
    _check_act("o", o, q.shape)
    _check_act("do", do, q.shape)
    _check_f32("lse", lse, (hq, total))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = int(library().cpattn_bwd_varlen_workspace_bytes(cu_p, nseq, hq, hkv, d, int(cp)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    rc = library().cpattn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), cu_p, nseq, hq, hkv, d, int(cp),
                                     1 if causal else 0, 0.0 if scale is None else float(scale),
                                     _stream_handle(stream, q, k, v, o, lse, do, dq, dk, dv, workspace))
    if rc:
        raise CpattnError(rc, "cpattn_bwd_varlen")
    return dq, dk, dv


def cpattn_bwd_workspace_bytes(b, s, hq, hkv, d, cp):
    return int(library().cpattn_bwd_workspace_bytes(b, s, hq, hkv, d, int(cp)))


def cpattn_bwd(q, k, v, o, lse, do, cp, causal=True, dq=None, dk=None, dv=None, workspace=None, stream=None,
               stage=None, scale=None):
    """Backward from the forward's saved o and lse. Returns (dq, dk, dv).

    ``stage`` (0, 1 or 2) runs only that stage of the backward (see
    cpattn_bwd_stage in include/cpattn.h); None runs all three. ``scale``:
    the forward's softmax scale when it was not 1/sqrt(d) (cpattn_bwd_ex;
    whole backward only).
    """
    b, s, hq, hkv, d = _dims(q, k, v)
    _check_act("o", o, q.shape)
    _check_act("do", do, q.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (b, hq, s) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [b, hq, s] tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_act("dq", dq, q.shape)
    _check_act("dk", dk, k.shape)
    _check_act("dv", dv, v.shape)
    need = cpattn_bwd_workspace_bytes(b, s, hq, hkv, d, cp)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    ws_bytes = workspace.numel() * workspace.element_size()
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), ws_bytes, b, s, hq, hkv, d, int(cp),
            1 if causal else 0, _stream_handle(stream, q, k, v, o, lse, do, dq, dk, dv, workspace))
    if scale is not None:
        if stage is not None:
            raise ValueError("a custom scale runs the whole backward (stage must be None)")
        rc = library().cpattn_bwd_ex(*ptrs[:-1], float(scale), ptrs[-1])
    elif stage is None:
        rc = library().cpattn_bwd(*ptrs)
    else:
        rc = library().cpattn_bwd_stage(int(stage), *ptrs)
    if rc:
        raise CpattnError(rc, "cpattn_bwd" if stage is None else "cpattn_bwd_stage")
    return dq, dk, dv


def _rank_dims(q, k, v, cp):
    """Shapes of a rank-local call: q [b, 2c, hq, d] (the rank's shard) and
    k, v [cp, b, 2c, hkv, d] (every rank's shard, rank-major) or [b, 2c, hkv, d]
    (one rank's shard). Returns b, s (the full sequence), hq, hkv, d."""
    _check_act("q", q)
    if q.dim() != 4:
        raise ValueError("q must be the rank's shard [b, 2c, hq, d]")
    b, local, hq, d = q.shape
    _check_act("k", k)
    _check_act("v", v, k.shape)
    shard = tuple(k.shape[-4:]) if k.dim() in (4, 5) else None
    if shard is None or shard[0] != b or shard[1] != local or shard[3] != d:
        raise ValueError("k and v must be [cp, b, 2c, hkv, d] or [b, 2c, hkv, d] matching q")
    if k.dim() == 5 and k.shape[0] != cp:
        raise ValueError(f"k and v hold {k.shape[0]} shards, expected cp = {cp}")
    return b, local * int(cp), hq, shard[2], d


def cpattn_fwd_rank(q, k_all, v_all, cp, rank, causal=True, scale=None, o=None, lse=None, stream=None):
    """One rank's forward in a CP group spread over GPUs (all-gather form).

    q: this rank's zigzag shard [b, 2c, hq, d] (chunk ``rank`` then chunk
    2cp-1-rank); k_all, v_all: every rank's shard [cp, b, 2c, hkv, d], as an
    all-gather leaves them. Runs every CP step of the rank in one launch with
    the merge on chip. Returns (o [b, 2c, hq, d] bf16, lse [b, hq, 2c] fp32).
    """
    if k_all.dim() != 5:
        raise ValueError("k_all and v_all must be [cp, b, 2c, hkv, d]")
    b, s, hq, hkv, d = _rank_dims(q, k_all, v_all, cp)
    local = q.shape[1]
    o = torch.empty_like(q) if o is None else o
    _check_act("o", o, q.shape)
    lse = torch.empty(b, hq, local, device=q.device, dtype=torch.float32) if lse is None else lse
    _check_f32("lse", lse, (b, hq, local))
    rc = library().cpattn_fwd_rank(q.data_ptr(), k_all.data_ptr(), v_all.data_ptr(), o.data_ptr(), lse.data_ptr(), b,
                                   s, hq, hkv, d, int(cp), int(rank), 1 if causal else 0,
                                   0.0 if scale is None else float(scale),
                                   _stream_handle(stream, q, k_all, v_all, o, lse))
    if rc:
        raise CpattnError(rc, "cpattn_fwd_rank")
    return o, lse


def cpattn_fwd_rank_step(q, k_blk, v_blk, cp, rank, step, causal=True, scale=None, o_part=None, lse_part=None,
                         stream=None):
    """One CP step of one rank (ring form): q is the rank's shard
    [b, 2c, hq, d], k_blk/v_blk the shard [b, 2c, hkv, d] of rank
    (rank - step) mod cp. Returns the step's unmerged result (o_part
    [b, 2c, hq, d] fp32, lse_part [b, hq, 2c]); rows outside the step get 0
    and -inf."""
    if k_blk.dim() != 4:
        raise ValueError("k_blk and v_blk must be one rank's shard [b, 2c, hkv, d]")
    b, s, hq, hkv, d = _rank_dims(q, k_blk, v_blk, cp)
    local = q.shape[1]
    if o_part is None:
        o_part = torch.empty(b, local, hq, d, device=q.device, dtype=torch.float32)
    if lse_part is None:
        lse_part = torch.empty(b, hq, local, device=q.device, dtype=torch.float32)
    _check_f32("o_part", o_part, (b, local, hq, d))
    _check_f32("lse_part", lse_part, (b, hq, local))
    rc = library().cpattn_fwd_rank_step(q.data_ptr(), k_blk.data_ptr(), v_blk.data_ptr(), o_part.data_ptr(),
                                        lse_part.data_ptr(), b, s, hq, hkv, d, int(cp), int(rank), int(step),
                                        1 if causal else 0, 0.0 if scale is None else float(scale),
                                        _stream_handle(stream, q, k_blk, v_blk, o_part, lse_part))
    if rc:
        raise CpattnError(rc, "cpattn_fwd_rank_step")
    return o_part, lse_part


def cpattn_bwd_rank_workspace_bytes(b, s, hq, hkv, d, cp):
    return int(library().cpattn_bwd_rank_workspace_bytes(b, s, hq, hkv, d, int(cp)))


def cpattn_bwd_rank(q, k_all, v_all, o, lse, do, cp, rank, causal=True, scale=None, dq=None, dk_part=None,
                    dv_part=None, workspace=None, stream=None, stage=None):
    """One rank's backward in a CP group spread over GPUs (all-gather form).

    q, o, do: the rank's shard [b, 2c, hq, d]; lse [b, hq, 2c]; k_all, v_all
    every rank's shard [cp, b, 2c, hkv, d]. Returns (dq [b, 2c, hq, d],
    dk_part, dv_part [cp, b, 2c, hkv, d]): the rank's own dQ, and its share
    of every rank's dK/dV, which a reduce-scatter over the group sums.
    ``stage`` (0, 1 or 2) runs only that stage (cpattn_bwd_rank_stage): the
    shares are complete after stage 1, dq after stage 2; stages share the
    workspace, which the caller then passes to each.
    """
    if k_all.dim() != 5:
        raise ValueError("k_all and v_all must be [cp, b, 2c, hkv, d]")
    b, s, hq, hkv, d = _rank_dims(q, k_all, v_all, cp)
    local = q.shape[1]
    _check_act("o", o, q.shape)
    _check_act("do", do, q.shape)
    _check_f32("lse", lse, (b, hq, local))
    dq = torch.empty_like(q) if dq is None else dq
    dk_part = torch.empty_like(k_all) if dk_part is None else dk_part
    dv_part = torch.empty_like(v_all) if dv_part is None else dv_part
    _check_act("dq", dq, q.shape)
    _check_act("dk_part", dk_part, k_all.shape)
    _check_act("dv_part", dv_part, v_all.shape)
    need = cpattn_bwd_rank_workspace_bytes(b, s, hq, hkv, d, cp)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    ptrs = (q.data_ptr(), k_all.data_ptr(), v_all.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
            dq.data_ptr(), dk_part.data_ptr(), dv_part.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), b, s, hq, hkv, d, int(cp), int(rank), 1 if causal else 0,
            0.0 if scale is None else float(scale),
            _stream_handle(stream, q, k_all, v_all, o, lse, do, dq, dk_part, dv_part, workspace))
    if stage is None:
        rc = library().cpattn_bwd_rank(*ptrs)
    else:
        rc = library().cpattn_bwd_rank_stage(int(stage), *ptrs)
    if rc:
        raise CpattnError(rc, "cpattn_bwd_rank" if stage is None else "cpattn_bwd_rank_stage")
    return dq, dk_part, dv_part


def cpattn_set_max_ctas(max_ctas):
    """Cap the persistent attention kernels' grid at max_ctas CTAs (one per
    SM; 0 = every SM), leaving the other SMs to kernels on other streams.
    Outputs are bit-identical for any cap. Process-wide."""
    rc = library().cpattn_set_max_ctas(int(max_ctas))
    if rc:
        raise CpattnError(rc, "cpattn_set_max_ctas")


def cpattn_zigzag_index(s, cp):
    """int64 [cp, 2c] (host): global token of virtual rank r's local position."""
    c = s // (2 * cp) if cp > 0 else 0
    out = torch.empty(max(cp, 0), 2 * c, dtype=torch.int64)
    rc = library().cpattn_zigzag_index(int(s), int(cp), ctypes.c_void_p(out.data_ptr()))
    if rc:
        raise CpattnError(rc, "cpattn_zigzag_index")
    return out


def cpattn_selftest_wait_timeout(limit_ns=10_000_000, stream=None):
    """Enqueue the self-test of the bounded waits: one wait that nothing
    completes gives up after ``limit_ns`` and sets bit 16 of the device status
    word (read it with cpattn_device_status)."""
    rc = library().cpattn_selftest_wait_timeout(int(limit_ns), _stream_handle(stream))
    if rc:
        raise CpattnError(rc, "cpattn_selftest_wait_timeout")


def cpattn_device_status(stream=None):
    """Read and clear the library's sticky device status word (0 = clean)."""
    st = ctypes.c_int(0)
    rc = library().cpattn_device_status(_stream_handle(stream), ctypes.byref(st))
    if rc not in (0, -7):
        raise CpattnError(rc, "cpattn_device_status")
    return int(st.value)

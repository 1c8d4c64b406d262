"""The allocation-free backward entry point, cpattn_bwd_noalloc.

It serves callers that cannot allocate device memory when they run the
backward (a device-memory budget fixed at start-up, threads that must not
enter an allocator, bindings without a device allocator) and so cannot pass
cpattn_bwd a workspace: it uses the library's fixed scratch array instead.
Here it is called through the C ABI and compared with cpattn_bwd (caller
workspace) on the same inputs, twice in a row. Both run the same
deterministic kernels, so the gradients must agree bit for bit (which is
within the backward's tolerance, relative L2 <= 2e-2, a fortiori). This
file is collected last.
"""
import ctypes

import pytest
import torch

from context_blockwise_causal_gb300 import cpattn_bwd, cpattn_device_status, cpattn_fwd, library
from context_blockwise_causal_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

REL_L2 = 2e-2


def _rel(x, ref):
    x, ref = x.double(), ref.double()
    return ((x - ref).norm() / ref.norm().clamp_min(1e-30)).item()


@pytest.mark.parametrize("b,s,hq,hkv,d,cp", [(1, 2048, 8, 2, 128, 4), (2, 960, 6, 2, 64, 3)])
def test_noalloc_matches_workspace_backward_twice(b, s, hq, hkv, d, cp):
    lib = library()
    w = Workload("noalloc", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, backward=True, seed=41 + s)
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], cp)
    ref = cpattn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], cp)
    torch.cuda.synchronize()
    assert lib.cpattn_bwd_workspace_bytes(b, s, hq, hkv, d, cp) <= lib.cpattn_bwd_noalloc_max_scratch_bytes()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        dq = torch.full_like(x["q"], float("nan"))
        dk = torch.full_like(x["k"], float("nan"))
        dv = torch.full_like(x["v"], float("nan"))
        rc = lib.cpattn_bwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), x["do"].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                    b, s, hq, hkv, d, cp, 1, stream)
        assert rc == 0, lib.cpattn_strerror(rc)
        torch.cuda.synchronize()
        assert cpattn_device_status() == 0
        for got, want in zip((dq, dk, dv), ref):
            assert torch.isfinite(got.float()).all()
            assert _rel(got.float(), want.float()) <= REL_L2
            assert torch.equal(got, want)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = library()
    cap = lib.cpattn_bwd_noalloc_max_scratch_bytes()
    b, s, hq, hkv, d, cp = 1, 131072, 128, 8, 128, 16
    assert lib.cpattn_bwd_workspace_bytes(b, s, hq, hkv, d, cp) > cap
    p = ctypes.c_void_p(4096)  # never dereferenced: the size check comes first
    rc = lib.cpattn_bwd_noalloc(p, p, p, p, p, p, p, p, p, b, s, hq, hkv, d, cp, 1, None)
    assert rc == -5  # CPATTN_ERR_WORKSPACE_TOO_SMALL

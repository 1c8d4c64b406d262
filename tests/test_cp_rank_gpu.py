"""The rank-local entry points (one rank's share of a CP group spread over
GPUs) through the C ABI, on one GPU: every rank of a group is run in turn on
this device, with its K/V exchange stood in for by local copies of the other
ranks' shards.

* Against the CPU fp64 oracle, every element: each rank's forward (the
  all-gather form, and the ring form through cp_group's own step-and-merge
  loop) equals the uncut attention's rows of that rank (max |O err| <= 1e-2
  beyond the bf16 output's half ulp, max |LSE err| <= 1e-3), and the sum over
  the ranks of their dK/dV shares -- rounded to bf16 after every addition, as
  a bf16 reduce-scatter may -- and each rank's dQ meet relative L2 <= 2e-2.
* Against the single-GPU kernels, bit for bit: a rank's forward, step
  results and dQ are those rows of cpattn_fwd / cpattn_fwd_step / cpattn_bwd
  (the same work units, computed the same way).
* The driver with a one-rank NCCL group: the collectives' code path on CUDA
  tensors, plain and checked (every collective fingerprinted).
"""
import datetime
import socket

import pytest
import torch

import oracle
from context_blockwise_causal_gb300 import (cpattn_bwd, cpattn_bwd_rank, cpattn_device_status, cpattn_fwd,
                                            cpattn_fwd_rank, cpattn_fwd_rank_step, cpattn_fwd_step)
from context_blockwise_causal_gb300.cp_group import CheckedExchange, cp_backward, cp_forward, zigzag_shard
from context_blockwise_causal_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, REL_L2 = 1e-2, 1e-3, 2e-2


def _half_ulp(x):
    ax = x.abs()
    e = torch.floor(torch.log2(torch.where(ax > 0, ax, torch.ones_like(ax))))
    return torch.where(ax > 0, torch.exp2(e - 8), torch.zeros_like(ax))


def _rel(x, ref):
    x, ref = x.double(), ref.double()
    return ((x - ref).norm() / ref.norm().clamp_min(1e-30)).item()


class LocalRing:
    """The ring exchange of one rank, on one GPU: at each hop the receive
    buffers get the next step's shard, copied from the other ranks' shards."""

    def __init__(self, k_shards, v_shards, rank):
        self.k, self.v, self.rank, self.cp, self.hop = k_shards, v_shards, rank, len(k_shards), 0

    def ring_start(self, send, recv, tag=None):
        self.hop += 1
        j = (self.rank - self.hop) % self.cp
        recv[0].copy_(self.k[j])
        recv[1].copy_(self.v[j])
        return None

    @staticmethod
    def ring_wait(reqs):
        pass


SMALL = [
    # b, s, hq, hkv, d, cp, causal
    (1, 1024, 4, 2, 128, 2, True),    # GQA, c = 256 (two tiles per chunk)
    (2, 960, 6, 2, 64, 3, True),      # batch 2, ragged chunks (c = 160), head pairs across groups
    (1, 1536, 4, 4, 128, 4, True),    # MHA, c = 192
    (1, 768, 3, 1, 128, 3, False),    # no mask, odd hq
    (1, 16, 2, 1, 64, 4, True),       # c = 2
]


@pytest.mark.parametrize("b,s,hq,hkv,d,cp,causal", SMALL)
def test_rank_local_forward_backward_all_elements(b, s, hq, hkv, d, cp, causal):
    w = Workload("rank", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, causal=causal, backward=True, seed=70 + s + cp)
    x = make_inputs(w, device="cuda")
    sh = {n: [zigzag_shard(t, cp, r) for r in range(cp)] for n, t in x.items()}
    k_all, v_all = torch.stack(sh["k"]), torch.stack(sh["v"])
    cpu = {n: t.cpu() for n, t in x.items()}
    o_ref, l_ref = oracle.attention_forward(cpu["q"], cpu["k"], cpu["v"], causal=causal)
    dq_ref, dk_ref, dv_ref = oracle.attention_backward(cpu["q"], cpu["k"], cpu["v"], cpu["do"], causal=causal)
    gidx = oracle.zigzag_global_index(s, cp)
    dk_sum = dv_sum = None
    for r in range(cp):
        rows = gidx[r]
        o_a, l_a = cpattn_fwd_rank(sh["q"][r], k_all, v_all, cp, r, causal=causal)
        o_r, l_r = cp_forward(sh["q"][r], sh["k"][r], sh["v"][r], causal=causal, form="ring",
                              exchange=LocalRing(sh["k"], sh["v"], r))
        dq, dk_p, dv_p = cpattn_bwd_rank(sh["q"][r], k_all, v_all, o_a, l_a, sh["do"][r], cp, r, causal=causal)
        torch.cuda.synchronize()
        assert cpattn_device_status() == 0
        for o, lse in ((o_a, l_a), (o_r, l_r)):
            err = (o.double().cpu() - o_ref[:, rows]).abs()
            assert (err - _half_ulp(o_ref[:, rows])).max().item() <= O_TOL, err.max().item()
            assert (lse.double().cpu() - l_ref[:, :, rows]).abs().max().item() <= LSE_TOL
        assert _rel(dq.float().cpu(), dq_ref[:, rows]) <= REL_L2
        # a bf16 reduce-scatter: the shares added one rank at a time, rounded to bf16 each time
        dk_sum = dk_p if dk_sum is None else (dk_sum.float() + dk_p.float()).to(torch.bfloat16)
        dv_sum = dv_p if dv_sum is None else (dv_sum.float() + dv_p.float()).to(torch.bfloat16)
    for r in range(cp):
        assert _rel(dk_sum[r].float().cpu(), zigzag_shard(dk_ref, cp, r)) <= REL_L2
        assert _rel(dv_sum[r].float().cpu(), zigzag_shard(dv_ref, cp, r)) <= REL_L2


@pytest.mark.parametrize("b,s,hq,hkv,d,cp", [(1, 8192, 8, 2, 128, 4), (2, 1920, 4, 1, 64, 3), (1, 4096, 6, 6, 128, 2)])
def test_rank_local_results_are_the_single_gpu_rows(b, s, hq, hkv, d, cp):
    """A rank runs exactly the single-GPU launch's work units for its rows, so
    its forward, its step results and its dQ are bit-identical to those rows
    of cpattn_fwd, cpattn_fwd_step and cpattn_bwd; its dK/dV shares sum to the
    single-GPU dK/dV within the backward's tolerance."""
    w = Workload("rank_bits", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, backward=True, seed=90 + s)
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], cp)
    dq, dk, dv = cpattn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], cp)
    steps = [cpattn_fwd_step(x["q"], x["k"], x["v"], cp, i) for i in range(cp)]
    sh = {n: [zigzag_shard(t, cp, r) for r in range(cp)] for n, t in x.items()}
    k_all, v_all = torch.stack(sh["k"]), torch.stack(sh["v"])
    dk_sum = torch.zeros(k_all.shape, device="cuda")
    dv_sum = torch.zeros(v_all.shape, device="cuda")
    for r in range(cp):
        o_r, l_r = cpattn_fwd_rank(sh["q"][r], k_all, v_all, cp, r)
        assert torch.equal(o_r, zigzag_shard(o, cp, r))
        assert torch.equal(l_r, zigzag_shard(lse, cp, r, dim=2))
        for i in range(cp):
            j = (r - i) % cp
            op, lp = cpattn_fwd_rank_step(sh["q"][r], sh["k"][j], sh["v"][j], cp, r, i)
            assert torch.equal(op, zigzag_shard(steps[i][0], cp, r)), (r, i)
            assert torch.equal(lp, zigzag_shard(steps[i][1], cp, r, dim=2)), (r, i)
        dq_r, dk_p, dv_p = cpattn_bwd_rank(sh["q"][r], k_all, v_all, o_r, l_r, sh["do"][r], cp, r)
        assert torch.equal(dq_r, zigzag_shard(dq, cp, r))
        dk_sum += dk_p.float()
        dv_sum += dv_p.float()
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    for r in range(cp):
        assert _rel(dk_sum[r], zigzag_shard(dk, cp, r).float()) <= REL_L2
        assert _rel(dv_sum[r], zigzag_shard(dv, cp, r).float()) <= REL_L2


def test_rank_local_argument_errors():
    from context_blockwise_causal_gb300 import library

    lib = library()
    p = torch.empty(1024, device="cuda")
    ptr = p.data_ptr()
    # rank outside [0, cp), and s not divisible by 2cp: rejected before any launch
    assert lib.cpattn_fwd_rank(ptr, ptr, ptr, ptr, ptr, 1, 256, 2, 2, 64, 2, 2, 1, 0.0, None) == -1
    assert lib.cpattn_fwd_rank(ptr, ptr, ptr, ptr, ptr, 1, 250, 2, 2, 64, 2, 0, 1, 0.0, None) == -1
    assert lib.cpattn_fwd_rank_step(ptr, ptr, ptr, ptr, ptr, 1, 256, 2, 2, 64, 2, 0, 2, 1, 0.0, None) == -1
    assert lib.cpattn_fwd_rank_step(ptr, ptr, ptr, ptr, ptr, 1, 256, 2, 2, 64, 2, -1, 0, 1, 0.0, None) == -1
    assert lib.cpattn_fwd_rank(ptr, ptr, ptr, ptr, ptr, 1, 256, 2, 2, 64, 2, 0, 1, -1.0, None) == -1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_driver_with_a_one_rank_nccl_group():
    """cp_forward (both forms) and cp_backward through a real NCCL process
    group of one rank: the collectives run on CUDA tensors, and with cp = 1
    the rank's results are the single-GPU kernels' bit for bit."""
    import torch.distributed as dist

    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120))
    try:
        w = Workload("nccl1", b=1, s=2048, hq=4, hkv=2, d=128, cp=1, backward=True, seed=5)
        x = make_inputs(w, device="cuda")
        o, lse = cpattn_fwd(x["q"], x["k"], x["v"], 1)
        dq, dk, dv = cpattn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], 1)
        o_a, l_a, k_all, v_all = cp_forward(x["q"], x["k"], x["v"], keep_kv=True)
        o_r, l_r = cp_forward(x["q"], x["k"], x["v"], form="ring")
        g = cp_backward(x["q"], x["k"], x["v"], o_a, l_a, x["do"], kv_all=(k_all, v_all))
        g2 = cp_backward(x["q"], x["k"], x["v"], o_a, l_a, x["do"])
        torch.cuda.synchronize()
        assert cpattn_device_status() == 0
        assert torch.equal(o_a, o) and torch.equal(l_a, lse)
        assert torch.equal(k_all[0], x["k"]) and torch.equal(v_all[0], x["v"])
        # the ring form's result comes through the fp32 step output and a conversion
        assert (o_r.float() - o.float()).abs().max().item() <= 2 * O_TOL
        assert (l_r - lse).abs().max().item() <= 2 * LSE_TOL
        for got in (g, g2):
            for a, b_ in zip(got, (dq, dk, dv)):
                assert torch.equal(a, b_)
        # the checked exchange: fingerprints and checksums of CUDA tensors
        # through NCCL, results unchanged
        ex = CheckedExchange()
        o_c, l_c = cp_forward(x["q"], x["k"], x["v"], exchange=ex)
        g3 = cp_backward(x["q"], x["k"], x["v"], o_c, l_c, x["do"], exchange=ex)
        torch.cuda.synchronize()
        assert torch.equal(o_c, o) and torch.equal(l_c, lse) and ex.sequence == 5
        for a, b_ in zip(g3, (dq, dk, dv)):
            assert torch.equal(a, b_)
    finally:
        dist.destroy_process_group()


def _random_rank_geometries(n, seed):
    """Half of them with odd head groups and an even number of tiles per
    chunk, where the forward pairs query tiles of one head."""
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        cp = rng.randint(2, 4)
        c = rng.randint(1, 300)
        b = rng.randint(1, 2)
        hkv = rng.randint(1, 2)
        hq = hkv * rng.randint(1, 4)
        tile_pairs = (hq // hkv) % 2 == 1 and ((c + 127) // 128) % 2 == 0
        if b * 2 * cp * c * hq > 8192 or tile_pairs != (len(out) % 2 == 0):
            continue
        out.append((b, 2 * cp * c, hq, hkv, rng.choice([64, 128]), cp, rng.random() < 0.75))
    return out


@pytest.mark.parametrize("b,s,hq,hkv,d,cp,causal", _random_rank_geometries(6, seed=23))
def test_rank_local_random_geometries_match_single_gpu_rows(b, s, hq, hkv, d, cp, causal):
    """Seeded random geometries (ragged chunks, head groups 1-4 -- tile pairs
    among them --, d 64/128, either mask): every rank's forward, step results
    and dQ bit for bit against the single-GPU launches' rows, its dK/dV shares
    summed over the ranks within the backward's tolerance."""
    w = Workload("rank_rand", b=b, s=s, hq=hq, hkv=hkv, d=d, cp=cp, causal=causal, backward=True, seed=s + 31 * hq)
    x = make_inputs(w, device="cuda")
    o, lse = cpattn_fwd(x["q"], x["k"], x["v"], cp, causal=causal)
    dq, dk, dv = cpattn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], cp, causal=causal)
    steps = [cpattn_fwd_step(x["q"], x["k"], x["v"], cp, i, causal=causal) for i in range(cp)]
    sh = {n: [zigzag_shard(t, cp, r) for r in range(cp)] for n, t in x.items()}
    k_all, v_all = torch.stack(sh["k"]), torch.stack(sh["v"])
    dk_sum = torch.zeros(k_all.shape, device="cuda")
    dv_sum = torch.zeros(v_all.shape, device="cuda")
    for r in range(cp):
        o_r, l_r = cpattn_fwd_rank(sh["q"][r], k_all, v_all, cp, r, causal=causal)
        assert torch.equal(o_r, zigzag_shard(o, cp, r)) and torch.equal(l_r, zigzag_shard(lse, cp, r, dim=2))
        for i in range(cp):
            j = (r - i) % cp
            op, lp = cpattn_fwd_rank_step(sh["q"][r], sh["k"][j], sh["v"][j], cp, r, i, causal=causal)
            assert torch.equal(op, zigzag_shard(steps[i][0], cp, r)) and torch.equal(
                lp, zigzag_shard(steps[i][1], cp, r, dim=2)), (r, i)
        dq_r, dk_p, dv_p = cpattn_bwd_rank(sh["q"][r], k_all, v_all, o_r, l_r, sh["do"][r], cp, r, causal=causal)
        assert torch.equal(dq_r, zigzag_shard(dq, cp, r))
        dk_sum += dk_p.float()
        dv_sum += dv_p.float()
    torch.cuda.synchronize()
    assert cpattn_device_status() == 0
    for r in range(cp):
        assert _rel(dk_sum[r], zigzag_shard(dk, cp, r).float()) <= REL_L2
        assert _rel(dv_sum[r], zigzag_shard(dv, cp, r).float()) <= REL_L2

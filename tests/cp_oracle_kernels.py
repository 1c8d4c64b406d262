"""CPU stand-ins for one CP rank's device work, for the multi-rank tests.

TEST INFRASTRUCTURE. The exchange logic of context_blockwise_causal_gb300.cp_group
(ring hops, all-gather, reduce-scatter) is checked with gloo ranks on the CPU,
where the library's CUDA kernels cannot run. Two stand-ins take their place:

* OracleKernels computes each rank's share in fp64 from the oracle's own
  primitives -- the rank's CP step plan, block attention and log-sum-exp
  merge ("大模型面试宝典 · Megatron-LM 篇", 3.2 steps 2-5, 3.4), and the plain
  backward -- so the merged result of a whole group can be compared with
  attention over the uncut sequence.
* RecordingKernels computes nothing: it records which K/V each call received
  and returns values whose sums are exact, so the test can check the
  exchange bit for bit.
"""
import torch

import oracle

_F64 = torch.float64


def _local_rows(ch, owner, cp, c):
    """Rows of global chunk ch in a shard of rank `owner` (chunk owner first)."""
    assert ch in (owner, 2 * cp - 1 - owner)
    start = 0 if ch == owner else c
    return torch.arange(start, start + c)


class OracleKernels:
    """One rank's device work in fp64 on the CPU (same signatures as
    cp_group.CudaKernels)."""

    @staticmethod
    def fwd_rank_step(q, k_blk, v_blk, cp, rank, step, causal, scale, o_part=None, lse_part=None):
        b, local, hq, d = q.shape
        c = local // 2
        G = hq // k_blk.shape[2]
        scale = oracle.softmax_scale(d) if scale is None else scale
        _i, j, q_ch, kv_ch, masked = oracle.cp_step_plan(rank, cp, causal)[step]
        qr = torch.cat([_local_rows(ch, rank, cp, c) for ch in q_ch])
        kr = torch.cat([_local_rows(ch, j, cp, c) for ch in kv_ch])
        qpos = torch.cat([torch.arange(ch * c, ch * c + c) for ch in q_ch])
        kpos = torch.cat([torch.arange(ch * c, ch * c + c) for ch in kv_ch])
        o = torch.zeros(b, local, hq, d, dtype=_F64)
        lse = torch.full((b, hq, local), float("-inf"), dtype=_F64)
        for bi in range(b):
            for h in range(hq):
                Oi, Li = oracle.block_attention(q[bi, qr, h].to(_F64), k_blk[bi, kr, h // G].to(_F64),
                                                v_blk[bi, kr, h // G].to(_F64), qpos, kpos, masked, scale)
                o[bi, qr, h] = Oi
                lse[bi, h, qr] = Li
        return o, lse

    @staticmethod
    def lse_merge(o_a, lse_a, o_b, lse_b, o_out, lse_out, o_final):
        b, local, hq, d = o_a.shape
        dst = o_final if o_out is False else o_out
        for bi in range(b):
            for h in range(hq):
                parts = [(o_a[bi, :, h], lse_a[bi, h])]
                if o_b is not None:
                    parts.append((o_b[bi, :, h], lse_b[bi, h]))
                O, L = oracle.lse_merge(parts)
                dst[bi, :, h] = O
                lse_out[bi, h] = L

    @staticmethod
    def new_output(q):
        return torch.empty(q.shape, dtype=_F64)

    @classmethod
    def fwd_rank(cls, q, k_all, v_all, cp, rank, causal, scale):
        o_acc, l_acc = cls.fwd_rank_step(q, k_all[rank], v_all[rank], cp, rank, 0, causal, scale)
        for i in range(1, cp):
            j = (rank - i) % cp
            o_i, l_i = cls.fwd_rank_step(q, k_all[j], v_all[j], cp, rank, i, causal, scale)
            cls.lse_merge(o_acc, l_acc, o_i, l_i, o_acc, l_acc, None)
        return o_acc, l_acc

    @classmethod
    def bwd_rank_shares(cls, q, k_all, v_all, o, lse, do, cp, rank, causal, scale):
        dq, dk_part, dv_part = cls.bwd_rank(q, k_all, v_all, o, lse, do, cp, rank, causal, scale)
        return dk_part, dv_part, dq

    @staticmethod
    def bwd_rank_dq(pending):
        return pending

    @staticmethod
    def bwd_rank(q, k_all, v_all, o, lse, do, cp, rank, causal, scale):
        """The rank's dQ, and its share of every shard's dK/dV: the plain
        backward over the whole sequence with q and dO zero outside the rank's
        rows (a row with zero dO has dP = 0 and D = 0, hence dS = 0, so it adds
        nothing to dK or dV)."""
        from context_blockwise_causal_gb300.cp_group import zigzag_shard, zigzag_unshard

        k_full = zigzag_unshard(list(k_all.to(_F64)))
        v_full = zigzag_unshard(list(v_all.to(_F64)))
        b, local, hq, d = q.shape
        s = local * cp
        zeros = torch.zeros(b, local, hq, d, dtype=_F64)
        q_full = zigzag_unshard([q.to(_F64) if r == rank else zeros for r in range(cp)])
        do_full = zigzag_unshard([do.to(_F64) if r == rank else zeros for r in range(cp)])
        idx = oracle.zigzag_global_index(s, cp)[rank]
        dq, dk, dv = oracle.attention_backward(q_full, k_full, v_full, do_full, causal=causal, dq_rows=idx,
                                               scale=scale)
        dk_part = torch.stack([zigzag_shard(dk, cp, r) for r in range(cp)])
        dv_part = torch.stack([zigzag_shard(dv, cp, r) for r in range(cp)])
        return dq, dk_part, dv_part


class RecordingKernels:
    """Records what each call receives; returns exactly summable values."""

    def __init__(self):
        self.steps = []     # (step, k_blk, v_blk) of each ring step, in call order
        self.gathered = []  # (k_all, v_all) handed to fwd_rank / bwd_rank
        self.merges = 0

    def fwd_rank_step(self, q, k_blk, v_blk, cp, rank, step, causal, scale, o_part=None, lse_part=None):
        self.steps.append((step, k_blk.clone(), v_blk.clone()))
        b, local, hq, d = q.shape
        return torch.zeros(b, local, hq, d, dtype=_F64), torch.zeros(b, hq, local, dtype=_F64)

    def lse_merge(self, o_a, lse_a, o_b, lse_b, o_out, lse_out, o_final):
        self.merges += 1

    def new_output(self, q):
        return torch.empty(q.shape, dtype=_F64)

    def fwd_rank(self, q, k_all, v_all, cp, rank, causal, scale):
        self.gathered.append((k_all.clone(), v_all.clone()))
        b, local, hq, d = q.shape
        return torch.zeros(b, local, hq, d, dtype=_F64), torch.zeros(b, hq, local, dtype=_F64)

    def bwd_rank_shares(self, q, k_all, v_all, o, lse, do, cp, rank, causal, scale):
        self.gathered.append((k_all.clone(), v_all.clone()))
        # share of shard j from rank r: 1000 * (r + 1) + j, small integers, so
        # the reduce-scatter's sum is exact in any float type
        parts = torch.stack([torch.full(k_all.shape[1:], 1000.0 * (rank + 1) + j, dtype=_F64) for j in range(cp)])
        return parts, -parts, torch.zeros(q.shape, dtype=_F64)

    @staticmethod
    def bwd_rank_dq(pending):
        return pending

"""Context parallelism over several GPUs: the exchange between CP ranks.

The pages run CP with one rank per device. Rank r of a group of cp ranks
holds its zigzag shard of q, k, v, dO: chunks r and 2cp-1-r of the
sequence's 2*cp chunks, concatenated ("大模型面试宝典 · Megatron-LM 篇", 3.2
step 1 and 3.4). Two ways of moving K/V between the ranks appear there, and
both are here:

* ring ("大模型面试宝典 · Megatron-LM 篇", 3.1 point 2, 3.2 steps 2-5): at step
  i every rank passes the K/V shard it holds to the next rank and receives
  the previous rank's, so that it holds rank (r - i) mod cp's shard at step
  i. Step i's attention runs while the next shard is in flight (3.2: steps
  2 and 3 run at the same time); each step's partial output is merged into
  the running result through its log-sum-exp (3.2 steps 4-5).
* all-gather ("超大规模集群下大语言模型训练实操指南", section "超长文本场景解决方案"):
  the forward all-gathers K/V and runs every step of the rank in one fused
  launch; the backward all-gathers K/V again and reduce-scatters each rank's
  share of dK/dV.

This module only moves data: sends, receives and collectives of the
process group (NCCL between GPUs). Every piece of arithmetic -- each step's
attention, the merges, the backward -- runs in the library's kernels
through the rank-local entry points (cpattn_fwd_rank, cpattn_fwd_rank_step,
cpattn_lse_merge, cpattn_bwd_rank). Buffers handed to those kernels are
always local to the calling GPU; nothing reads another GPU's memory
directly.

The ``kernels`` and ``exchange`` arguments exist so that the exchange logic
can be checked on its own: tests pass recording or CPU stand-ins. The
default kernels are the CUDA library's, and it fails loudly when that
library is missing. ``exchange=CheckedExchange(group)`` fingerprints every
collective across the ranks (a debugging aid, see its docstring).

The attention kernels take a whole SM per CTA, so a send/receive kernel of
the communication library runs during a ring step only on SMs they leave
free: cpattn_set_max_ctas caps their grid (outputs unchanged).
"""
import zlib

import torch
import torch.distributed as dist

from . import cpattn_bwd_rank, cpattn_bwd_rank_workspace_bytes, cpattn_fwd_rank, cpattn_fwd_rank_step, cpattn_lse_merge

__all__ = ["CudaKernels", "GroupExchange", "CheckedExchange", "ExchangeMismatch", "zigzag_shard", "zigzag_unshard",
           "cp_forward", "cp_backward"]


class CudaKernels:
    """The device work of one rank: the library's rank-local entry points."""

    @staticmethod
    def fwd_rank(q, k_all, v_all, cp, rank, causal, scale):
        return cpattn_fwd_rank(q, k_all, v_all, cp, rank, causal=causal, scale=scale)

    @staticmethod
    def fwd_rank_step(q, k_blk, v_blk, cp, rank, step, causal, scale, o_part=None, lse_part=None):
        return cpattn_fwd_rank_step(q, k_blk, v_blk, cp, rank, step, causal=causal, scale=scale, o_part=o_part,
                                    lse_part=lse_part)

    @staticmethod
    def lse_merge(o_a, lse_a, o_b, lse_b, o_out, lse_out, o_final):
        """Merge (o_b, lse_b) into (o_a, lse_a); o_out=False writes the final
        bf16 output into o_final instead of an fp32 result."""
        cpattn_lse_merge(o_a, lse_a, o_b, lse_b, o_out=o_out, lse_out=lse_out, o_bf16=o_final)

    @staticmethod
    def new_output(q):
        return torch.empty_like(q)

    @staticmethod
    def bwd_rank_shares(q, k_all, v_all, o, lse, do, cp, rank, causal, scale):
        """The backward's first two stages: the rank's shares of every shard's
        dK/dV. Returns (dk_part, dv_part, pending); bwd_rank_dq(pending) then
        runs the dQ stage."""
        b, local, hq, d = q.shape
        ws = torch.empty(max(cpattn_bwd_rank_workspace_bytes(b, local * cp, hq, k_all.shape[3], d, cp), 16),
                         dtype=torch.uint8, device=q.device)
        dq, dk_part, dv_part = torch.empty_like(q), torch.empty_like(k_all), torch.empty_like(v_all)
        call = (q, k_all, v_all, o, lse, do, cp, rank)
        kw = dict(causal=causal, scale=scale, dq=dq, dk_part=dk_part, dv_part=dv_part, workspace=ws)
        for stage in (0, 1):
            cpattn_bwd_rank(*call, stage=stage, **kw)
        return dk_part, dv_part, (call, kw)

    @staticmethod
    def bwd_rank_dq(pending):
        call, kw = pending
        return cpattn_bwd_rank(*call, stage=2, **kw)[0]


class GroupExchange:
    """K/V movement between the ranks of a torch.distributed process group."""

    def __init__(self, group=None):
        self.group = group
        self.rank = dist.get_rank(group)
        self.cp = dist.get_world_size(group)
        # the ring: receive from the previous rank, send to the next
        self.next = self._global((self.rank + 1) % self.cp)
        self.prev = self._global((self.rank - 1) % self.cp)

    def _global(self, r):
        return r if self.group is None else dist.get_global_rank(self.group, r)

    def all_gather(self, x, tag=None):
        """Every rank's x stacked rank-major: [cp, *x.shape]. ``tag`` names
        the logical tensor (used by CheckedExchange)."""
        x = x.contiguous()
        # gathered as the concatenation along dimension 0 (the form every
        # backend takes), then viewed rank-major
        out = torch.empty((self.cp * x.shape[0],) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
        dist.all_gather_into_tensor(out, x, group=self.group)
        return out.view((self.cp,) + tuple(x.shape))

    def reduce_scatter_start(self, *parts, tag=None):
        """For each tensor of parts, [cp, *shape] on every rank, start summing
        over the ranks so that this rank gets the sum of their parts[rank].
        Returns a handle for reduce_scatter_finish; the reduction runs while
        the caller issues more work."""
        outs, works = [], []
        for p_ in parts:
            out = torch.empty(tuple(p_.shape[1:]), dtype=p_.dtype, device=p_.device)
            flat = p_.contiguous().view((p_.shape[0] * p_.shape[1],) + tuple(p_.shape[2:]))
            works.append(dist.reduce_scatter_tensor(out, flat, op=dist.ReduceOp.SUM, group=self.group, async_op=True))
            outs.append(out)
        return outs, works

    @staticmethod
    def reduce_scatter_finish(handle):
        outs, works = handle
        for w_ in works:
            w_.wait()
        return outs

    def ring_start(self, send, recv, tag=None):
        """Post one ring hop: each tensor of ``send`` goes to the next rank,
        each of ``recv`` is filled from the previous one. Returns the
        requests; the send and receive pairs are issued together, so no
        rank blocks on a send before its own receive is posted."""
        ops = [dist.P2POp(dist.isend, t, self.next, group=self.group) for t in send]
        ops += [dist.P2POp(dist.irecv, t, self.prev, group=self.group) for t in recv]
        return dist.batch_isend_irecv(ops)

    @staticmethod
    def ring_wait(reqs):
        for r in reqs or ():
            r.wait()


class ExchangeMismatch(RuntimeError):
    """The ranks of a CheckedExchange disagreed on a collective, or received
    bytes that differ from what their peer sent."""


_OPS = {"all_gather": 1, "reduce_scatter": 2, "ring": 3}
_DTYPES = (torch.bfloat16, torch.float16, torch.float32, torch.float64, torch.int64, torch.int32, torch.int16)
_MAX_TENSORS, _MAX_DIMS = 4, 6
_FIELDS = ("sequence", "operation", "logical id", "dimensions") + tuple(f"size {i}" for i in range(_MAX_DIMS)) + (
    "dtype", "checksum")


def _checksum(t):
    """A position-weighted sum of the tensor's 16-bit words, modulo 2^64
    (integer arithmetic, so every rank gets the same value for the same
    bytes). A debugging checksum, not part of any attention step."""
    w = t.detach().contiguous().view(-1).view(torch.int16).to(torch.int64) & 0xFFFF
    pos = torch.arange(w.numel(), dtype=torch.int64, device=w.device) % 65521 + 1
    return int((w * pos).sum().item())


class CheckedExchange(GroupExchange):
    """GroupExchange that fingerprints every logical collective.

    Page "Megatron 面试题（一）：模型抽象与训练数据流", item M024 (follow-up):
    collectives of the same shape issued in a different order on some rank
    can complete and give finite but wrong results, so each logical
    collective records its group, sequence number, operation, shape, dtype
    and an input checksum, and business tensors a logical id; comparing the
    records across ranks shows the first point where they diverge.

    Here, before each collective every rank all-gathers a fixed-size record
    (sequence number, operation, the caller's tag as logical id, and per
    tensor its shape, dtype and checksum). All ranks must agree on
    everything but the checksums; each rank sees every record, so on a
    mismatch every rank raises ExchangeMismatch before the collective itself
    runs, and none is left waiting in it. After an all-gather each rank's
    block is checked against its owner's checksum, after a ring hop the
    received tensors against the sender's; the ranks then agree (one more
    small all-gather) so that a failure on one raises on all. The checks add
    two small collectives and a pass over the data per collective: a
    debugging aid, off unless a caller passes this exchange.
    """

    def __init__(self, group=None):
        super().__init__(group)
        self.sequence = 0

    def _record(self, op, tag, tensors):
        if len(tensors) > _MAX_TENSORS:
            raise ValueError(f"at most {_MAX_TENSORS} tensors per checked collective")
        rows = []
        for t in tensors:
            if t.dim() > _MAX_DIMS or t.dtype not in _DTYPES:
                raise ValueError("tensor outside the checked exchange's shapes or dtypes")
            rows.append([self.sequence, _OPS[op], zlib.crc32(str(tag).encode()), t.dim()]
                        + list(t.shape) + [-1] * (_MAX_DIMS - t.dim()) + [_DTYPES.index(t.dtype), _checksum(t)])
        rows += [[self.sequence, _OPS[op], zlib.crc32(str(tag).encode())] + [-2] * (len(_FIELDS) - 3)] * (
            _MAX_TENSORS - len(tensors))
        dev = tensors[0].device if tensors else torch.device("cpu")
        mine = torch.tensor(rows, dtype=torch.int64, device=dev)
        every = torch.empty((self.cp * _MAX_TENSORS, len(_FIELDS)), dtype=torch.int64, device=dev)
        dist.all_gather_into_tensor(every, mine, group=self.group)
        every = every.view(self.cp, _MAX_TENSORS, len(_FIELDS)).cpu()
        meta = every[:, :, :-1]
        if not bool((meta == meta[0]).all()):
            r = int((meta != meta[0]).flatten(1).any(1).nonzero()[0])
            ti, fi = [int(x) for x in (meta[r] != meta[0]).nonzero()[0]]
            raise ExchangeMismatch(
                f"collective #{self.sequence} ({op} {tag!r}): rank {r} differs from rank 0 in the "
                f"{_FIELDS[fi]} of tensor {ti} ({int(meta[r, ti, fi])} against {int(meta[0, ti, fi])})")
        self.sequence += 1
        return every[:, :, -1]  # checksums [rank, tensor]

    def _agree(self, ok, what, dev):
        flags = torch.empty(self.cp, dtype=torch.int64, device=dev)
        dist.all_gather_into_tensor(flags, torch.tensor([0 if ok else 1], dtype=torch.int64, device=dev),
                                    group=self.group)
        bad = [r for r, f in enumerate(flags.cpu().tolist()) if f]
        if bad:
            raise ExchangeMismatch(f"{what}: received bytes differ from those sent on rank(s) {bad}")

    def all_gather(self, x, tag=None):
        sums = self._record("all_gather", tag, [x])
        out = super().all_gather(x, tag)
        ok = all(_checksum(out[r]) == int(sums[r, 0]) for r in range(self.cp))
        self._agree(ok, f"all_gather {tag!r}", x.device)
        return out

    def reduce_scatter_start(self, *parts, tag=None):
        self._record("reduce_scatter", tag, list(parts))
        return super().reduce_scatter_start(*parts, tag=tag)

    def ring_start(self, send, recv, tag=None):
        sums = self._record("ring", tag, list(send))
        return (super().ring_start(send, recv, tag), recv, sums[(self.rank - 1) % self.cp], tag)

    def ring_wait(self, handle):
        if handle is None:
            return
        GroupExchange.ring_wait(handle[0])
        self._verify_ring(handle)

    def _verify_ring(self, handle):
        _, recv, sums, tag = handle
        ok = all(_checksum(t) == int(sums[i]) for i, t in enumerate(recv))
        self._agree(ok, f"ring hop {tag!r}", recv[0].device)


def zigzag_shard(x, cp, rank, dim=1):
    """Rank ``rank``'s zigzag shard of a natural-order tensor: chunks rank and
    2cp-1-rank of dimension ``dim`` (length s, cut into 2cp chunks),
    concatenated. Data preparation for callers that start from whole
    sequences (a data loader normally hands each rank its shard)."""
    s = x.shape[dim]
    if s % (2 * cp):
        raise ValueError(f"length {s} is not divisible by 2*cp = {2 * cp}")
    c = s // (2 * cp)
    lo = x.narrow(dim, rank * c, c)
    hi = x.narrow(dim, (2 * cp - 1 - rank) * c, c)
    return torch.cat((lo, hi), dim=dim)


def zigzag_unshard(shards, dim=1):
    """Inverse of zigzag_shard: the natural-order tensor from every rank's
    shard (a list in rank order)."""
    cp = len(shards)
    c = shards[0].shape[dim] // 2
    chunks = [None] * (2 * cp)
    for r, sh in enumerate(shards):
        chunks[r] = sh.narrow(dim, 0, c)
        chunks[2 * cp - 1 - r] = sh.narrow(dim, c, c)
    return torch.cat(chunks, dim=dim)


def _ring_forward(q, k, v, rank, cp, causal, scale, kernels, exchange):
    # Two receive buffers alternate; the caller's own k, v serve step 0 and
    # are never written. A buffer is refilled only after the step that read
    # it was issued and its outgoing copy completed.
    recv = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(min(cp - 1, 2))]
    kv = (k, v)
    o = kernels.new_output(q)
    o_acc = l_acc = o_part = l_part = lse = None
    for i in range(cp):
        nxt = recv[i % 2] if i + 1 < cp else None
        reqs = exchange.ring_start(kv, nxt, tag=f"kv hop {i + 1}") if nxt is not None else None  # during step i
        if i == 0:
            o_acc, l_acc = kernels.fwd_rank_step(q, kv[0], kv[1], cp, rank, 0, causal, scale)
        else:
            o_part, l_part = kernels.fwd_rank_step(q, kv[0], kv[1], cp, rank, i, causal, scale, o_part, l_part)
        if i == cp - 1:
            # the last correction writes the bf16 output and the final lse
            lse = torch.empty_like(l_acc)
            kernels.lse_merge(o_acc, l_acc, o_part, l_part, False, lse, o)
        elif i > 0:
            kernels.lse_merge(o_acc, l_acc, o_part, l_part, o_acc, l_acc, None)
        exchange.ring_wait(reqs)
        if nxt is not None:
            kv = nxt
    return o, lse


def cp_forward(q, k, v, group=None, causal=True, scale=None, form="allgather", kernels=None, exchange=None,
               keep_kv=False):
    """CP attention forward of this rank. q [b, 2c, hq, d], k, v [b, 2c, hkv, d]:
    the rank's zigzag shards. Returns (o [b, 2c, hq, d], lse [b, hq, 2c]) for
    the rank's rows, equal to those rows of attention over the whole
    sequence; with ``keep_kv`` (all-gather form) also the gathered
    (k_all, v_all), which cp_backward can reuse instead of gathering again.

    form="allgather": one all-gather of K and of V, then every CP step in one
    fused launch (the merge on chip). form="ring": cp steps, each computed
    while the next shard travels one hop, merged step by step.
    """
    exchange = exchange or GroupExchange(group)
    kernels = kernels or CudaKernels
    rank, cp = exchange.rank, exchange.cp
    if form == "ring":
        if keep_kv:
            raise ValueError("keep_kv applies to the all-gather form")
        return _ring_forward(q, k, v, rank, cp, causal, scale, kernels, exchange)
    if form != "allgather":
        raise ValueError("form must be 'allgather' or 'ring'")
    k_all = exchange.all_gather(k, tag="k")
    v_all = exchange.all_gather(v, tag="v")
    o, lse = kernels.fwd_rank(q, k_all, v_all, cp, rank, causal, scale)
    return (o, lse, k_all, v_all) if keep_kv else (o, lse)


def cp_backward(q, k, v, o, lse, do, group=None, causal=True, scale=None, kv_all=None, kernels=None,
                exchange=None):
    """CP attention backward of this rank from its saved o and lse: all-gather
    K and V (unless ``kv_all`` = (k_all, v_all) from cp_forward is given),
    the rank's dK/dV kernels, then a reduce-scatter that sums every rank's
    share of each shard's dK/dV -- running while the rank's dQ kernel
    computes. Returns (dq, dk, dv) of the rank's shards."""
    exchange = exchange or GroupExchange(group)
    kernels = kernels or CudaKernels
    rank, cp = exchange.rank, exchange.cp
    if kv_all is None:
        kv_all = (exchange.all_gather(k, tag="k"), exchange.all_gather(v, tag="v"))
    dk_part, dv_part, pending = kernels.bwd_rank_shares(q, kv_all[0], kv_all[1], o, lse, do, cp, rank, causal, scale)
    handle = exchange.reduce_scatter_start(dk_part, dv_part, tag="dk dv")
    dq = kernels.bwd_rank_dq(pending)
    dk, dv = exchange.reduce_scatter_finish(handle)
    return dq, dk, dv

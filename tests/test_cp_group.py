"""The exchange between CP ranks (context_blockwise_causal_gb300.cp_group),
checked with gloo process groups of 2 and 3 ranks on the CPU.

* Ring form ("大模型面试宝典 · Megatron-LM 篇", 3.2 step 3): at step i rank r
  must compute with exactly the K/V shard of rank (r - i) mod cp, bit for
  bit, steps in order 0..cp-1, merging cp-1 times.
* All-gather form ("超大规模集群下大语言模型训练实操指南", 超长文本场景解决方案):
  the gathered K/V is every rank's shard in rank order, bit for bit; the
  reduce-scatter hands rank r the sum of every rank's share of shard r.
* End to end with the oracle's fp64 stand-ins for the kernels: each rank's
  forward (both forms) and backward equal the uncut oracle's rows within
  1e-12, and the shards are the zigzag map's rows.
* The checked exchange ("Megatron 面试题（一）：模型抽象与训练数据流", M024
  follow-up: a fingerprint of every logical collective): it leaves results
  bit-identical, and every rank raises together when one rank issues the
  collectives in another order, passes another shape, or receives bytes
  other than those sent (faults made on the host).
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(b, s, hq, hkv, d, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    mk = lambda h: torch.randn(b, s, h, d, generator=g).to(torch.bfloat16).to(dtype)  # noqa: E731
    return mk(hq), mk(hkv), mk(hkv), mk(hq)


def _worker(rank, world, port, case, fails):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case(rank, world)
    except Exception as e:  # reported to the parent
        import traceback

        fails[rank] = "".join(traceback.format_exception(e))[-3000:]
    finally:
        dist.destroy_process_group()


def _run(case, world):
    with mp.Manager() as m:
        fails = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), case, fails), nprocs=world, join=True)
        assert not dict(fails), "\n".join(dict(fails).values())


# ---------------------------------------------------------------- cases
def _ring_delivers_each_steps_shard(rank, cp):
    from cp_oracle_kernels import RecordingKernels

    from context_blockwise_causal_gb300.cp_group import cp_forward, zigzag_shard

    q, k, v, _ = _inputs(2, 24 * cp, 2, 1, 8, seed=11, dtype=torch.bfloat16)
    rec = RecordingKernels()
    kr, vr = zigzag_shard(k, cp, rank), zigzag_shard(v, cp, rank)
    cp_forward(zigzag_shard(q, cp, rank), kr, vr, form="ring", kernels=rec)
    assert [st for st, _, _ in rec.steps] == list(range(cp))
    for step, kb, vb in rec.steps:
        j = (rank - step) % cp
        assert torch.equal(kb, zigzag_shard(k, cp, j)) and torch.equal(vb, zigzag_shard(v, cp, j)), (step, j)
    # cp - 1 corrections, the last one writing the output (cp = 1: one conversion)
    assert rec.merges == max(cp - 1, 1)
    # the caller's shards are not overwritten by the receives
    assert torch.equal(kr, zigzag_shard(k, cp, rank)) and torch.equal(vr, zigzag_shard(v, cp, rank))


def _allgather_and_reduce_scatter_exact(rank, cp):
    from cp_oracle_kernels import RecordingKernels

    from context_blockwise_causal_gb300.cp_group import cp_backward, cp_forward, zigzag_shard

    q, k, v, do = _inputs(1, 16 * cp, 4, 2, 8, seed=12, dtype=torch.bfloat16)
    rec = RecordingKernels()
    sh = lambda x: zigzag_shard(x, cp, rank)  # noqa: E731
    cp_forward(sh(q), sh(k), sh(v), form="allgather", kernels=rec)
    _, dk, dv = cp_backward(sh(q), sh(k), sh(v), None, None, sh(do), kernels=rec)
    want_k = torch.stack([zigzag_shard(k, cp, r) for r in range(cp)])
    want_v = torch.stack([zigzag_shard(v, cp, r) for r in range(cp)])
    assert len(rec.gathered) == 2
    for k_all, v_all in rec.gathered:
        assert torch.equal(k_all, want_k) and torch.equal(v_all, want_v)
    # share of shard `rank` from rank r is 1000 (r + 1) + rank
    total = sum(1000.0 * (r + 1) + rank for r in range(cp))
    assert torch.equal(dk, torch.full_like(dk, total)) and torch.equal(dv, torch.full_like(dv, -total))


def _oracle_group_matches_uncut(rank, cp):
    import oracle
    from cp_oracle_kernels import OracleKernels

    from context_blockwise_causal_gb300.cp_group import cp_backward, cp_forward, zigzag_shard

    for causal, (b, c, hq, hkv, d) in ((True, (2, 5, 4, 2, 8)), (False, (1, 3, 3, 1, 4))):
        s = 2 * cp * c
        q, k, v, do = _inputs(b, s, hq, hkv, d, seed=13 + s, dtype=torch.float64)
        sh = lambda x: zigzag_shard(x, cp, rank)  # noqa: E731
        rows = oracle.zigzag_global_index(s, cp)[rank]
        o_ref, l_ref = oracle.attention_forward(q, k, v, causal=causal, rows=rows)
        for form in ("ring", "allgather"):
            o, lse = cp_forward(sh(q), sh(k), sh(v), causal=causal, form=form, kernels=OracleKernels)
            assert (o - o_ref).abs().max().item() <= 1e-12, (form, causal)
            assert (lse - l_ref).abs().max().item() <= 1e-12, (form, causal)
        o, lse = cp_forward(sh(q), sh(k), sh(v), causal=causal, kernels=OracleKernels)
        dq, dk, dv = cp_backward(sh(q), sh(k), sh(v), o, lse, sh(do), causal=causal, kernels=OracleKernels)
        dq_ref, dk_ref, dv_ref = oracle.attention_backward(q, k, v, do, causal=causal)
        assert (dq - dq_ref[:, rows]).abs().max().item() <= 1e-12
        assert (dk - zigzag_shard(dk_ref, cp, rank)).abs().max().item() <= 1e-12
        assert (dv - zigzag_shard(dv_ref, cp, rank)).abs().max().item() <= 1e-12


def _checked_exchange_changes_nothing(rank, cp):
    from cp_oracle_kernels import OracleKernels

    from context_blockwise_causal_gb300.cp_group import CheckedExchange, cp_backward, cp_forward, zigzag_shard

    b, c, hq, hkv, d = 1, 4, 4, 2, 8
    q, k, v, do = _inputs(b, 2 * cp * c, hq, hkv, d, seed=14, dtype=torch.float64)
    sh = lambda x: zigzag_shard(x, cp, rank)  # noqa: E731
    ex = CheckedExchange()
    for form in ("ring", "allgather"):
        plain = cp_forward(sh(q), sh(k), sh(v), form=form, kernels=OracleKernels)
        checked = cp_forward(sh(q), sh(k), sh(v), form=form, kernels=OracleKernels, exchange=ex)
        assert all(torch.equal(a, b_) for a, b_ in zip(plain, checked)), form
    o, lse = plain
    grads = cp_backward(sh(q), sh(k), sh(v), o, lse, sh(do), kernels=OracleKernels)
    grads_c = cp_backward(sh(q), sh(k), sh(v), o, lse, sh(do), kernels=OracleKernels, exchange=ex)
    assert all(torch.equal(a, b_) for a, b_ in zip(grads, grads_c))
    # ring: cp - 1 hops; all-gather forward: 2; backward: 2 gathers + 1 reduce-scatter
    assert ex.sequence == (cp - 1) + 2 + 3


def _checked_exchange_catches_order_swap(rank, cp):
    from context_blockwise_causal_gb300.cp_group import CheckedExchange, ExchangeMismatch

    ex = CheckedExchange()
    k = torch.full((2, 3), float(rank), dtype=torch.bfloat16)
    v = torch.full((2, 3), 10.0 + rank, dtype=torch.bfloat16)
    # same shapes and dtypes: without the check the gathers would complete
    # and mix K and V; rank 1 issues them in the other order
    order = [("k", k), ("v", v)] if rank == 0 else [("v", v), ("k", k)]
    with pytest.raises(ExchangeMismatch, match="logical id"):
        ex.all_gather(order[0][1], tag=order[0][0])


def _checked_exchange_catches_shape(rank, cp):
    from context_blockwise_causal_gb300.cp_group import CheckedExchange, ExchangeMismatch

    ex = CheckedExchange()
    x = torch.zeros(2, 3 + (rank == cp - 1), dtype=torch.bfloat16)
    with pytest.raises(ExchangeMismatch, match=f"rank {cp - 1} differs from rank 0 in the size 1"):
        ex.all_gather(x, tag="k")


def _checked_exchange_catches_corrupt_hop(rank, cp):
    from cp_oracle_kernels import RecordingKernels

    from context_blockwise_causal_gb300.cp_group import (CheckedExchange, ExchangeMismatch, GroupExchange, cp_forward,
                                                         zigzag_shard)

    class CorruptsOnRank0(CheckedExchange):
        # the hop completes, then rank 0's received K changes in one element
        # (a transfer fault made on the host) before the check
        def ring_wait(self, handle):
            if handle is None:
                return
            GroupExchange.ring_wait(handle[0])
            if self.rank == 0:
                handle[1][0].view(-1)[0] += 1
            self._verify_ring(handle)

    q, k, v, _ = _inputs(1, 8 * cp, 2, 1, 8, seed=15, dtype=torch.bfloat16)
    sh = lambda x: zigzag_shard(x, cp, rank)  # noqa: E731
    with pytest.raises(ExchangeMismatch, match=r"ring hop 'kv hop 1'.*rank\(s\) \[0\]"):
        cp_forward(sh(q), sh(k), sh(v), form="ring", kernels=RecordingKernels(), exchange=CorruptsOnRank0())


def _rank_leaves_worker(rank, world, port, out):
    # rank 1 leaves between steps (its process ends without entering the
    # exchange); rank 0's next collective must end in an error, not wait
    import datetime

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=10))
    if rank == 1:
        dist.destroy_process_group()
        return
    from cp_oracle_kernels import RecordingKernels

    from context_blockwise_causal_gb300.cp_group import cp_forward, zigzag_shard

    q, k, v, _ = _inputs(1, 8 * world, 2, 1, 8, seed=16, dtype=torch.bfloat16)
    sh = lambda x: zigzag_shard(x, world, rank)  # noqa: E731
    import time

    t0 = time.time()
    try:
        cp_forward(sh(q), sh(k), sh(v), form="allgather", kernels=RecordingKernels())
        out[rank] = "returned"
    except Exception as e:  # the collective reports the lost peer
        out[rank] = f"raised {type(e).__name__} after {time.time() - t0:.1f} s"
    finally:
        try:
            dist.destroy_process_group()
        except Exception:
            pass


@pytest.mark.timeout(120)
def test_a_rank_that_leaves_ends_the_others_collective_with_an_error():
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_leaves_worker, args=(2, _free_port(), out), nprocs=2, join=True)
        got = dict(out)
    assert got[0].startswith("raised"), got


@pytest.mark.parametrize("world", [2, 3])
def test_checked_exchange_changes_nothing(world):
    _run(_checked_exchange_changes_nothing, world)


@pytest.mark.parametrize("case", [_checked_exchange_catches_order_swap, _checked_exchange_catches_shape,
                                  _checked_exchange_catches_corrupt_hop])
def test_checked_exchange_raises_on_every_rank(case):
    _run(case, 2)


@pytest.mark.parametrize("world", [2, 3])
def test_ring_delivers_each_steps_shard(world):
    _run(_ring_delivers_each_steps_shard, world)


@pytest.mark.parametrize("world", [2, 3])
def test_allgather_and_reduce_scatter_are_exact(world):
    _run(_allgather_and_reduce_scatter_exact, world)


@pytest.mark.parametrize("world", [2, 3])
def test_group_with_oracle_kernels_matches_uncut_attention(world):
    _run(_oracle_group_matches_uncut, world)


def test_single_rank_group_ring_is_one_step():
    _run(_ring_delivers_each_steps_shard, 1)


def test_zigzag_shard_round_trip_matches_the_map():
    import oracle

    from context_blockwise_causal_gb300.cp_group import zigzag_shard, zigzag_unshard

    x = torch.arange(2 * 48 * 3).reshape(2, 48, 3)
    for cp in (1, 2, 3, 4, 6):
        shards = [zigzag_shard(x, cp, r) for r in range(cp)]
        assert torch.equal(zigzag_unshard(shards), x)
        gidx = oracle.zigzag_global_index(48, cp)
        for r in range(cp):
            assert torch.equal(shards[r], x[:, gidx[r]])

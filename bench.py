"""Benchmark: context-parallel causal attention forward + backward on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
cpattn_fwd (all virtual CP ranks, fused LSE merge) then the three stages of
cpattn_bwd (row vectors, dK/dV, dQ), through the C-ABI library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an
independent replica of the workload on its own GPU: the method needs no
exchange on one GPU, so there is no collective on the data path; value is the
work of all ranks divided by the slowest rank's time ("scaling": "weak").
--impl reference times the CPU fp64 oracle on a bounded sample of the same
workload on the host cores (the reference arm of the comparison).
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CP causal attention fwd/bwd TFLOP/s and % of GB300 dense BF16 peak"
DEFAULT_WORKLOAD = "train_b1_s32768_h32kv8_d128_cp8"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def _max_over_ranks(value, device, ws):
    """The largest of `value` over the ranks of the default process group
    (the slowest rank sets the job's time); `value` itself when alone."""
    if ws <= 1:
        return float(value)
    import torch.distributed as dist

    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # let nvidia-smi initialise before the timed region starts
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0:
                time.sleep(0.02)
            self.lines.clear()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons, masks = [], None, set(), set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            masks.add(f[4])
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [x for x in sm if smax is None or x > 0.3 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "active_reason_masks": sorted(masks), "samples": len(sm)}


def _profile_traffic(kernel_file, profile_name):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel (same sha256); else None."""
    prof = os.path.join(ROOT, "profiles", profile_name)
    src = os.path.join(ROOT, "context_blockwise_causal_gb300", "csrc", kernel_file)
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    text = open(prof).read()
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_b and m_h):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != m_h.group(1):
        return None
    return float(m_b.group(1))


# ------------------------------------------------------------------ CPU oracle arm
_CPU_INPUTS = {}


def _oracle_sample(w, rows_n, seed):
    """The CPU oracle on a bounded sample of workload w: forward O/LSE and the
    backward's dQ for `rows_n` seeded random query rows of every head.
    Returns (seconds, algorithmic FLOPs of what the sample computes: per
    visible (query, key) pair, 2*d for each of the five products it forms --
    S and P.V for the forward, then S again, dP = dO.V^T and dS.K for dQ)."""
    import oracle
    from context_blockwise_causal_gb300.workloads import make_inputs, sample_rows

    if w.name not in _CPU_INPUTS:
        _CPU_INPUTS[w.name] = make_inputs(w, device="cpu")
    x = _CPU_INPUTS[w.name]
    rows = sample_rows(w, rows_n, seed=seed)
    t0 = time.perf_counter()
    oracle.attention_forward(x["q"], x["k"], x["v"], causal=w.causal, rows=rows, row_block=256)
    oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], causal=w.causal, dq_rows=rows, dkv_heads=[],
                              row_block=256)
    dt = time.perf_counter() - t0
    keys = (rows + 1).double().sum().item() if w.causal else float(w.s) * rows.numel()
    flops = 5 * 2.0 * w.d * keys * w.hq * w.b
    return dt, flops


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    cores = torch.get_num_threads()
    # about 4096 sampled rows over the whole run (32..1024 per step), so the
    # run stays within a few minutes whatever --steps is, unless given
    rows_n = args.ref_rows or max(32, min(1024, 4096 // (args.steps + args.warmup)))
    for _ in range(args.warmup):
        _oracle_sample(w, rows_n, seed=w.seed + 5)
    times, flops = [], 0.0
    for i in range(args.steps):
        dt, fl = _oracle_sample(w, rows_n, seed=w.seed + 5)
        times.append(dt)
        flops = fl
    tot = sum(times)
    value = flops * args.steps / tot / 1e12
    sample = (f"{rows_n} seeded query rows x {w.hq} heads of {w.name}: forward O/LSE + backward dQ "
              f"(CPU fp64 oracle, torch float64 on {cores} threads)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def _config(w, n):
    return {"workload": w.name, "b": w.b, "s": w.s, "hq": w.hq, "hkv": w.hkv, "d": w.d, "cp": w.cp,
            "causal": w.causal, "step": "cpattn_fwd + cpattn_bwd",
            "l2": f"inputs larger than L2 (q,k,v,dO = {_in_bytes(w) / 1e6:.0f} MB > 129 MB)",
            "parallelism": "replicas" if n > 1 else "single"}


def _in_bytes(w):
    return 2 * (2 * w.b * w.s * w.hq * w.d + 2 * w.b * w.s * w.hkv * w.d)


def run_ours(args, w):
    import torch.distributed as dist

    from context_blockwise_causal_gb300 import (cpattn_bwd, cpattn_bwd_workspace_bytes, cpattn_device_status,
                                                cpattn_fwd, library)
    from context_blockwise_causal_gb300.workloads import make_inputs

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl")
    library()
    dev = torch.device("cuda", local)
    x = make_inputs(w, device=dev, seed=w.seed + rank)
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o = torch.empty_like(q)
    lse = torch.empty(w.b, w.hq, w.s, device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsp = torch.empty(cpattn_bwd_workspace_bytes(w.b, w.s, w.hq, w.hkv, w.d, w.cp), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = 4  # forward; backward row vectors, dK/dV, dQ

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(evs=None):
        # one event before the forward and after each kernel: the forward,
        # then the backward's three stages (row vectors, dK/dV, dQ)
        if evs:
            evs[0].record(stream)
        cpattn_fwd(q, k, v, w.cp, causal=w.causal, o=o, lse=lse, stream=stream)
        if evs:
            evs[1].record(stream)
        for stage in range(3):
            cpattn_bwd(q, k, v, o, lse, do, w.cp, causal=w.causal, dq=dq, dk=dk, dv=dv, workspace=wsp,
                       stream=stream, stage=stage)
            if evs:
                evs[2 + stage].record(stream)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    if cpattn_device_status(stream) != 0:
        raise RuntimeError("a kernel reported a timeout during warm-up")

    # ---- device-timed region: inputs resident in HBM
    evs = [[ev() for _ in range(5)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        t_start, t_end = ev(), ev()
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        barrier()
    total_ms = t_start.elapsed_time(t_end)
    kern_ms = {name: sum(e[i].elapsed_time(e[i + 1]) for e in evs) / len(evs)
               for i, name in enumerate(("fwd", "bwd_pre", "bwd_dkdv", "bwd_dq"))}
    if cpattn_device_status(stream) != 0:
        raise RuntimeError("a kernel reported a timeout in the timed region")
    total_ms = _max_over_ranks(total_ms, dev, ws)

    # ---- end to end through the public API with host buffers: every step
    # copies its inputs in from pinned host memory and its gradients out to
    # pinned host memory. The copies run on their own streams (one each way)
    # with two device buffer sets, so step i+1's inputs arrive and step i's
    # gradients leave while kernels run, as a prefetching training loop does;
    # every step's copies lie inside the timed region. Both start once the
    # forward of the step they overlap has finished: the forward keeps K/V
    # tiles in L2 and slows most when copy traffic passes through it.
    pin = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "do")}
    out_h = {n: torch.empty(tuple(tt.shape), dtype=tt.dtype).pin_memory() for n, tt in (("dq", dq), ("dk", dk), ("dv", dv))}
    h2d = sum(tt.numel() * tt.element_size() for tt in pin.values())
    d2h = sum(tt.numel() * tt.element_size() for tt in out_h.values())
    bufs = [dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv)]
    bufs.append({n: torch.empty_like(t) for n, t in bufs[0].items()})
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def fwd_on(B):
        cpattn_fwd(B["q"], B["k"], B["v"], w.cp, causal=w.causal, o=B["o"], lse=B["lse"], stream=stream)

    def bwd_on(B):
        for stage in range(3):
            cpattn_bwd(B["q"], B["k"], B["v"], B["o"], B["lse"], B["do"], w.cp, causal=w.causal, dq=B["dq"],
                       dk=B["dk"], dv=B["dv"], workspace=wsp, stream=stream, stage=stage)

    def e2e_run(nsteps):
        computed = [None, None]  # per buffer set: its last step's kernels are done
        copied = [None, None]    # per buffer set: its last step's gradients are on the host

        def copy_in(i, after):
            B = bufs[i % 2]
            if computed[i % 2] is not None:
                s_in.wait_event(computed[i % 2])  # step i-2 no longer reads these inputs
            if after is not None:
                s_in.wait_event(after)
            with torch.cuda.stream(s_in):
                for n in ("q", "k", "v", "do"):
                    B[n].copy_(pin[n], non_blocking=True)
            e = ev()
            e.record(s_in)
            return e

        def copy_out(B, done, after):
            s_out.wait_event(done)
            if after is not None:
                s_out.wait_event(after)
            with torch.cuda.stream(s_out):
                for n in ("dq", "dk", "dv"):
                    out_h[n].copy_(B[n], non_blocking=True)
            e = ev()
            e.record(s_out)
            return e

        start = ev()
        start.record(s_in)
        arrived = copy_in(0, None)
        pending = None  # the previous step's gradients, sent once this step's forward is done
        for i in range(nsteps):
            B = bufs[i % 2]
            stream.wait_event(arrived)
            if copied[i % 2] is not None:
                stream.wait_event(copied[i % 2])  # step i-2's gradients have left
            fwd_on(B)
            fwd_done = ev()
            fwd_done.record(stream)
            if pending is not None:
                copied[pending[2] % 2] = copy_out(pending[0], pending[1], fwd_done)
                pending = None
            bwd_on(B)
            done = ev()
            done.record(stream)
            computed[i % 2] = done
            if i + 1 < nsteps:
                arrived = copy_in(i + 1, fwd_done)
                pending = (B, done, i)
            else:
                copied[i % 2] = copy_out(B, done, None)
        end = ev()
        end.record(s_out)
        return start, end

    e2e_run(2)
    with ClockSampler(local) as clk_e2e:
        barrier()
        e0, e1 = e2e_run(args.steps)
        barrier()
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), dev, ws)
    del bufs[1]

    # ---- the unfused forward (cp step launches + cp-1 merges), outside the
    # timed step: the baseline the fused forward is measured against
    unfused = None
    if not args.no_unfused:
        from context_blockwise_causal_gb300 import cpattn_fwd_unfused, cpattn_fwd_unfused_workspace_bytes

        uws = torch.empty(cpattn_fwd_unfused_workspace_bytes(w.b, w.s, w.hq, w.d), dtype=torch.uint8, device=dev)
        o_u = torch.empty_like(q)
        lse_u = torch.empty_like(lse)
        for _ in range(2):
            cpattn_fwd_unfused(q, k, v, w.cp, causal=w.causal, o=o_u, lse=lse_u, workspace=uws, stream=stream)
        barrier()
        u0, u1 = ev(), ev()
        u0.record(stream)
        for _ in range(args.steps):
            cpattn_fwd_unfused(q, k, v, w.cp, causal=w.causal, o=o_u, lse=lse_u, workspace=uws, stream=stream)
        u1.record(stream)
        barrier()
        if cpattn_device_status(stream) != 0:
            raise RuntimeError("a kernel reported a timeout in the unfused forward")
        u_ms = u0.elapsed_time(u1) / args.steps
        # one merge on its own (HBM-bound): read two fp32 O and LSE, write one
        from context_blockwise_causal_gb300 import cpattn_lse_merge

        nb = w.b * w.s * w.hq * w.d * 4
        o_a = uws[:nb].view(torch.float32).view(w.b, w.s, w.hq, w.d)
        o_b = uws[nb:2 * nb].view(torch.float32).view(w.b, w.s, w.hq, w.d)
        o_a.zero_()
        o_b.zero_()
        l_a = torch.zeros_like(lse)
        l_b = torch.zeros_like(lse)
        cpattn_lse_merge(o_a, l_a, o_b, l_b, o_out=o_a, lse_out=l_a, stream=stream)
        barrier()
        m0, m1 = ev(), ev()
        m0.record(stream)
        for _ in range(args.steps):
            cpattn_lse_merge(o_a, l_a, o_b, l_b, o_out=o_a, lse_out=l_a, stream=stream)
        m1.record(stream)
        barrier()
        m_ms = m0.elapsed_time(m1) / args.steps
        m_bytes = 3 * nb + 3 * lse.numel() * 4
        unfused = {"ms": u_ms, "tflops": w.fwd_flops() / (u_ms * 1e-3) / 1e12,
                   "launches_per_call": 2 * w.cp - 1 if w.cp > 1 else 2,
                   "fused_fwd_ms": kern_ms["fwd"], "unfused_over_fused": u_ms / kern_ms["fwd"],
                   "merge": {"ms": m_ms, "bytes": m_bytes, "gbs": m_bytes / (m_ms * 1e-3) / 1e9,
                             "hbm_frac": m_bytes / (m_ms * 1e-3) / 1e9 / _peaks()["hbm_gbs"]}}
        del uws, o_a, o_b

    # ---- RoPE of q and k in place (HBM-bound), forward then inverse
    from context_blockwise_causal_gb300 import cpattn_rope

    for inv in (False, True):
        cpattn_rope(q, inverse=inv, stream=stream)
        cpattn_rope(k, inverse=inv, stream=stream)
    barrier()
    r0, r1 = ev(), ev()
    r0.record(stream)
    for i in range(2 * args.steps):
        cpattn_rope(q, inverse=bool(i & 1), stream=stream)
        cpattn_rope(k, inverse=bool(i & 1), stream=stream)
    r1.record(stream)
    barrier()
    rope_ms = r0.elapsed_time(r1) / (2 * args.steps)
    rope_bytes = 2 * (q.numel() + k.numel()) * 2  # read and write q and k, bf16
    rope = {"ms": rope_ms, "bytes": rope_bytes, "gbs": rope_bytes / (rope_ms * 1e-3) / 1e9,
            "what": "cpattn_rope on q and k (two launches)"}

    # ---- packed samples of the same total length (attention within samples):
    # a mix of long samples, and many short ones; one launch per kernel
    from context_blockwise_causal_gb300 import cpattn_bwd_varlen, cpattn_fwd_varlen

    qp, kp, vp, dop = (t[0].reshape(w.s, t.shape[2], w.d) for t in (q, k, v, do))

    def packed(lens):
        cu = [0]
        for n_ in lens:
            cu.append(cu[-1] + n_)
        o_p, lse_p = cpattn_fwd_varlen(qp, kp, vp, cu, w.cp, stream=stream)
        g_p = cpattn_bwd_varlen(qp, kp, vp, o_p, lse_p, dop, cu, w.cp, stream=stream)
        barrier()
        va, vb, vc = ev(), ev(), ev()
        va.record(stream)
        for _ in range(args.steps):
            cpattn_fwd_varlen(qp, kp, vp, cu, w.cp, o=o_p, lse=lse_p, stream=stream)
        vb.record(stream)
        for _ in range(args.steps):
            cpattn_bwd_varlen(qp, kp, vp, o_p, lse_p, dop, cu, w.cp, dq=g_p[0], dk=g_p[1], dv=g_p[2], stream=stream)
        vc.record(stream)
        barrier()
        if cpattn_device_status(stream) != 0:
            raise RuntimeError("a kernel reported a timeout in the packed-sample run")
        vf_ms, vbw_ms = va.elapsed_time(vb) / args.steps, vb.elapsed_time(vc) / args.steps
        fl = sum(2.0 * w.hq * n_ * n_ * w.d for n_ in lens)
        return {"samples": lens if len(lens) <= 8 else f"{len(lens)} x {lens[0]}", "fwd_ms": vf_ms, "bwd_ms": vbw_ms,
                "fwd_tflops": fl / (vf_ms * 1e-3) / 1e12, "bwd_tflops": 2.5 * fl / (vbw_ms * 1e-3) / 1e12,
                "launches": {"fwd": 1, "bwd": 3}}

    varlen = {"mixed": packed([w.s // 2, w.s // 4, w.s // 8, w.s // 16, w.s // 16]),
              "short": packed([2048] * (w.s // 2048))}

    # ---- one CP group spread over GPUs, its compute side on this GPU: each
    # rank's forward (all-gather form) and backward on its shard, one rank
    # after another; the slowest rank bounds a group step. No exchange is
    # timed (one GPU here); the all-gathered K/V are built locally.
    cp_ranks = None
    if not args.no_cp_ranks and w.cp > 1:
        from context_blockwise_causal_gb300 import cpattn_bwd_rank, cpattn_fwd_rank
        from context_blockwise_causal_gb300.cp_group import zigzag_shard

        sh = {n: [zigzag_shard(t, w.cp, r) for r in range(w.cp)] for n, t in (("q", q), ("k", k), ("v", v), ("do", do))}
        k_all, v_all = torch.stack(sh["k"]), torch.stack(sh["v"])
        per = []
        for r in range(w.cp):
            o_r, l_r = cpattn_fwd_rank(sh["q"][r], k_all, v_all, w.cp, r, causal=w.causal, stream=stream)
            g_r = cpattn_bwd_rank(sh["q"][r], k_all, v_all, o_r, l_r, sh["do"][r], w.cp, r, causal=w.causal,
                                  stream=stream)
            tf, tb = [], []
            for _ in range(3):
                e0c, e1c, e2c = ev(), ev(), ev()
                e0c.record(stream)
                cpattn_fwd_rank(sh["q"][r], k_all, v_all, w.cp, r, causal=w.causal, o=o_r, lse=l_r, stream=stream)
                e1c.record(stream)
                cpattn_bwd_rank(sh["q"][r], k_all, v_all, o_r, l_r, sh["do"][r], w.cp, r, causal=w.causal,
                                dq=g_r[0], dk_part=g_r[1], dv_part=g_r[2], stream=stream)
                e2c.record(stream)
                e2c.synchronize()
                tf.append(e0c.elapsed_time(e1c))
                tb.append(e1c.elapsed_time(e2c))
            per.append({"rank": r, "fwd_ms": statistics.median(tf), "bwd_ms": statistics.median(tb)})
        if cpattn_device_status(stream) != 0:
            raise RuntimeError("a kernel reported a timeout in the per-rank run")
        mf = max(p_["fwd_ms"] for p_ in per)
        mb = max(p_["bwd_ms"] for p_ in per)
        cp_ranks = {"ranks": w.cp, "per_rank": per, "max_fwd_ms": mf, "max_bwd_ms": mb,
                    "compute_scaling": {"fwd": kern_ms["fwd"] / w.cp / mf,
                                        "bwd": (kern_ms["bwd_pre"] + kern_ms["bwd_dkdv"] + kern_ms["bwd_dq"]) / w.cp / mb},
                    "what": "each rank's cpattn_fwd_rank and cpattn_bwd_rank on its zigzag shard with every rank's "
                            "K/V gathered locally, on this one GPU; compute_scaling = (fused single-GPU time / cp) / "
                            "slowest rank's time; the K/V exchange is not timed"}
        del sh, k_all, v_all

    # ---- the forward on the other configurations (each: warm-up, then the
    # median of several launches, L2 flushed before each)
    sweep = {}
    if not args.no_sweep and rank == 0:
        from context_blockwise_causal_gb300.workloads import WORKLOADS, make_inputs as _mk
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        for name, cw in WORKLOADS.items():
            if name == w.name or name.startswith("train_"):
                continue
            xi = _mk(cw, device=dev, with_grad=False)
            o_c, lse_c = cpattn_fwd(xi["q"], xi["k"], xi["v"], cw.cp, causal=cw.causal, stream=stream)
            reps = 3 if cw.fwd_flops() > 5e13 else 10
            tms = []
            for _ in range(reps):
                with torch.cuda.stream(stream):
                    flush.zero_()
                e0c, e1c = ev(), ev()
                e0c.record(stream)
                cpattn_fwd(xi["q"], xi["k"], xi["v"], cw.cp, causal=cw.causal, o=o_c, lse=lse_c, stream=stream)
                e1c.record(stream)
                e1c.synchronize()
                tms.append(e0c.elapsed_time(e1c))
            if cpattn_device_status(stream) != 0:
                raise RuntimeError(f"a kernel reported a timeout in the {name} forward")
            ms = statistics.median(tms)
            sweep[name] = {"fwd_ms": ms, "fwd_tflops": cw.fwd_flops() / (ms * 1e-3) / 1e12, "reps": reps}
            del xi, o_c, lse_c
        del flush

    if rank == 0:
        peaks = _peaks()
        step_flops = w.fwd_flops() + w.bwd_flops()
        value = step_flops * args.steps * ws / (total_ms * 1e-3) / 1e12
        fwd_avg = kern_ms["fwd"]
        bwd_avg = kern_ms["bwd_pre"] + kern_ms["bwd_dkdv"] + kern_ms["bwd_dq"]
        fwd_tf = w.fwd_flops() / (fwd_avg * 1e-3) / 1e12
        bwd_tf = w.bwd_flops() / (bwd_avg * 1e-3) / 1e12
        # per-kernel algorithmic work: the matmuls each tensor-bound kernel
        # performs (forward 2, dK/dV 4, dQ 3 -- S and dP are formed in both
        # backward kernels), bytes for the HBM-bound preprocess
        kern_flops = {"fwd": w.fwd_flops(), "bwd_dkdv": 2.0 * w.fwd_flops(), "bwd_dq": 1.5 * w.fwd_flops()}
        pre_bytes = 2 * 2 * w.b * w.s * w.hq * w.d + 4 * w.b * w.hq * w.s * 3
        dominant = max(kern_flops, key=lambda n: kern_ms[n])
        achieved = kern_flops[dominant] / (kern_ms[dominant] * 1e-3) / 1e12
        # the step lasts tens of milliseconds, so its kernels are measured
        # against the burst peak (the sustained one is for seconds-long loops)
        peak = peaks["bf16_tflops"]
        src = {"fwd": ("fwd_kernel.cuh", "cpattn_fwd_kernel"), "bwd_dkdv": ("bwd_kernel.cuh", "cpattn_bwd_dkdv_kernel"),
               "bwd_dq": ("bwd_kernel.cuh", "cpattn_bwd_dq_kernel")}[dominant]
        traffic = _profile_traffic(src[0], f"{src[1]}_{w.name}.md")
        kernels = {n: {"ms": kern_ms[n], "tflops": kern_flops[n] / (kern_ms[n] * 1e-3) / 1e12} for n in kern_flops}
        kernels["bwd_pre"] = {"ms": kern_ms["bwd_pre"], "gbs": pre_bytes / (kern_ms["bwd_pre"] * 1e-3) / 1e9,
                              "hbm_frac": pre_bytes / (kern_ms["bwd_pre"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _config(w, ws),
            "fraction_of_peak": {"vs_burst": value / ws / peaks["bf16_tflops"],
                                 "vs_sustained": value / ws / peaks["bf16_tflops_sustained"],
                                 "peaks": peaks["source"]},
            "phases": {"fwd_ms": fwd_avg, "fwd_tflops": fwd_tf, "fwd_frac_burst": fwd_tf / peaks["bf16_tflops"],
                       "bwd_ms": bwd_avg, "bwd_tflops": bwd_tf, "bwd_frac_burst": bwd_tf / peaks["bf16_tflops"],
                       "flops": {"fwd": w.fwd_flops(), "bwd": w.bwd_flops(), "convention": "fwd 2*b*hq*s^2*d; bwd 2.5x fwd"}},
            "kernels": kernels,
            "roofline": {"kernel": src[1], "bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "peak_kind": f"bf16 burst ({peaks['source']})",
                         "frac_vs_sustained": achieved / peaks["bf16_tflops_sustained"], "traffic": traffic,
                         "flops_per_launch": kern_flops[dominant]},
            "e2e": {"value": step_flops * args.steps * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps,
                    "copies": "pinned host <-> device every step, on two copy streams overlapping the backward "
                              "kernels (started after each forward; two device buffer sets)",
                    "clocks": clk_e2e.summary()},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
        }
        if unfused is not None:
            line["unfused_fwd"] = unfused
        rope["hbm_frac"] = rope["gbs"] / peaks["hbm_gbs"]
        line["rope"] = rope
        line["varlen"] = varlen
        if cp_ranks is not None:
            line["cp_ranks"] = cp_ranks
        if sweep:
            for v_ in sweep.values():
                v_["frac_burst"] = v_["fwd_tflops"] / peaks["bf16_tflops"]
                v_["frac_sustained"] = v_["fwd_tflops"] / peaks["bf16_tflops_sustained"]
            line["fwd_other_configs"] = sweep
        if not args.no_cpu_baseline:
            ref_rows = args.ref_rows or 1024
            dt, fl = _oracle_sample(w, ref_rows, seed=w.seed + 5)
            line["cpu_baseline"] = {
                "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": torch.get_num_threads(), "kind": "oracle",
                "sample": f"{ref_rows} seeded query rows x {w.hq} heads of {w.name}: forward O/LSE + backward "
                          f"dQ (CPU fp64 oracle), {dt:.1f} s"}
            # the same oracle on one thread, on a smaller sample of the same rows' kind
            nthr = torch.get_num_threads()
            torch.set_num_threads(1)
            try:
                rows1 = max(1, ref_rows // 16)
                dt1, fl1 = _oracle_sample(w, rows1, seed=w.seed + 6)
            finally:
                torch.set_num_threads(nthr)
            line["cpu_baseline"]["single_thread"] = {"value": fl1 / dt1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                                                     "sample": f"{rows1} seeded query rows, {dt1:.1f} s"}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--ref-rows", type=int, default=None,
                    help="oracle rows per sample (default: 1024 for the CPU baseline; the reference arm spreads "
                         "about 4096 rows over its steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true", help="skip timing the unfused forward")
    ap.add_argument("--no-sweep", action="store_true", help="skip the forward on the other configurations")
    ap.add_argument("--no-cp-ranks", action="store_true",
                    help="skip timing each CP rank's share of the workload (the multi-GPU form's compute)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    from context_blockwise_causal_gb300.workloads import WORKLOADS

    w = WORKLOADS[args.workload]
    if not w.backward:
        raise SystemExit("the bench step is forward + backward: pick a workload with a backward")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

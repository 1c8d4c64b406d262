"""Host-side tests of bench.py that need no GPU: the reference arm (the CPU
oracle timed on a bounded sample) prints the contract's JSON line, alone and
under torchrun with two ranks (rank 0 alone reports), and the max-over-ranks
reduction of the timed region works across two gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
ARGS = ["--impl", "reference", "--workload", "small_b1_s512_h4_d64_cp2", "--steps", "1", "--warmup", "3",
        "--ref-rows", "16"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(out):
    return [json.loads(ln) for ln in out.splitlines() if ln.startswith("{")]


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", *ARGS], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    ln = lines[0]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in ln, key
    assert ln["impl"] == "reference" and ln["value"] > 0 and ln["unit"] == "TFLOP/s"
    assert ln["cpu_baseline"]["kind"] == "oracle" and ln["cpu_baseline"]["cores"] >= 1
    assert ln["e2e"]["h2d_bytes_per_step"] == 0 and ln["e2e"]["value"] == ln["value"]


def test_reference_arm_under_torchrun_reports_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--gpus", "2", *ARGS]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def _rank_main(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    sys.path.insert(0, ROOT)
    import bench

    got = bench._max_over_ranks(10.0 + 5 * rank, torch.device("cpu"), 2)
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_timed_region_takes_the_slowest_rank_gloo():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(port, out), nprocs=2, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}
    import bench  # single process: the value itself

    assert bench._max_over_ranks(3.5, torch.device("cpu"), 1) == 3.5



def test_profile_traffic_only_for_the_current_kernel_source(tmp_path, monkeypatch):
    """bench.py reports a kernel's DRAM traffic from its committed ncu summary
    only when the summary was taken on the kernel source as it is now (the
    sha256 in the summary matches); otherwise traffic is null."""
    import hashlib

    import bench

    src_dir = tmp_path / "context_blockwise_causal_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = src_dir / "k.cuh"
    src.write_bytes(b"__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles" / "k_w.md").write_text(f"kernel_source_sha256: {sha}\ndram_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._profile_traffic("k.cuh", "k_w.md") == 12345.0
    src.write_bytes(b"__global__ void k() { }\n")  # the kernel changed since the capture
    assert bench._profile_traffic("k.cuh", "k_w.md") is None
    assert bench._profile_traffic("k.cuh", "missing.md") is None

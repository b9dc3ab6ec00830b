"""The N > 1 host path on CPU with gloo, world size 2.

The hot path needs no exchange between GPUs: each rank runs a replica of the whole step on its
own batch, and the job's time is the slowest rank's.  What needs checking without GPUs is that
host logic: the max over ranks, the whole-job throughput, and that under torchrun only rank 0
prints the bench line (the reference arm, which runs on the host cores, shows it end to end).
"""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest
import torch
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    import torch.distributed as dist
    sys.path.insert(0, str(ROOT))
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.5 + 2.0 * rank, "cpu")      # rank 0: 1.5 ms, rank 1: 3.5 ms
        value = bench.replica_throughput(world, 256, ms)
        Path(outdir, f"r{rank}.json").write_text(json.dumps({"ms": ms, "value": value}))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [json.loads(Path(tmp_path, f"r{r}.json").read_text()) for r in range(2)]
    for g in got:
        assert g["ms"] == 3.5                                   # every rank sees the slowest
        assert g["value"] == pytest.approx(2 * 256 / 3.5e-3)    # both replicas' tokens over that time


def test_single_process_is_identity():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks(2.25, "cpu") == 2.25
    assert bench.replica_throughput(1, 100, 1000.0) == pytest.approx(100.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), str(ROOT / "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny_bf16", "--steps", "1", "--warmup", "3",
           "--cpu-tokens", "8"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["config"]["workload"] == "tiny_bf16"
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"

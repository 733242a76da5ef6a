"""The multi-rank path of bench.py on CPU (gloo, world size 2).

The attention has no exchange step, so N GPUs run N independent replicas: the
only cross-rank traffic is the barrier around the timed region and the maximum
of the ranks' times, and the reported value is all ranks' work over that
maximum.  These tests run that host logic in two gloo processes, and the
reference arm of the benchmark under torchrun with two ranks (rank 0 alone
runs and prints).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, lr = bench.rank_info()
    assert (r, w, lr) == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = [12.5, 40.0][rank]          # rank 1 is the slow replica
    dist.barrier()
    ms = bench.max_over_ranks(my_ms, dist, "cpu")
    value = bench.whole_job_tflops(world, 1e15, 4, ms)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo(tmp_path):
    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    # both ranks see the slowest rank's time, and the value counts both replicas' work
    assert res[0] == res[1]
    assert res[0]["ms"] == 40.0
    assert res[0]["value"] == pytest.approx(2 * 1e15 * 4 / 0.040 / 1e12)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(7.0, None, "cpu") == 7.0
    assert bench.whole_job_tflops(1, 2e12, 10, 1000.0) == pytest.approx(20.0)   # 2e13 FLOP in 1 s


def test_reference_arm_under_torchrun_prints_one_line():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "3", "--warmup", "3",
           "--ref-rows", "16"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"

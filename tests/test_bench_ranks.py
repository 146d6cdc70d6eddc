"""The benchmark's N > 1 path on the CPU: world-size-2 gloo process groups.

The path does not shard across GPUs by a collective: every rank runs the same
workload (replicas, weak scaling), the job's time is the slowest rank's, and
the job's throughput is world x one rank's work over that time. These tests
run the rank helpers of bench.py in two processes over gloo, and launch the
CPU reference arm under torchrun with two ranks, where rank 0 alone runs the
oracle and prints the line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.rank_env() == (world, rank, rank)
        # rank r took (10 + r) ms for the device steps and (30 - r) ms end to end
        ms, e2e = bench.max_over_ranks([10.0 + rank, 30.0 - rank], world)
        value = bench.job_tflops(world, 2.0e12, 5, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "e2e": e2e, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_gloo(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:  # every rank agrees on the slowest rank's times
        assert r["ms"] == 11.0 and r["e2e"] == 30.0
        # two replicas of 5 steps of 2e12 FLOP in 11 ms
        assert r["value"] == pytest.approx(2 * 2.0e12 * 5 / 11.0e-3 / 1e12)


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.job_tflops(1, 1.0e12, 1, 1.0) == pytest.approx(1000.0)


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once(tmp_path):
    """Two ranks launched the way the benchmark driver launches N > 1: rank 0
    times the oracle and prints one JSON line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"

"""The N > 1 host path of bench.py on CPU, with the gloo backend (no GPU needed).

Every rank runs its own replica of the workload (heads and batch items are
independent, so the path has no exchange step); the only cross-rank traffic is
timing: the job's time is the slowest rank's, and the job's throughput counts the
units of every replica.  The reference arm (the CPU oracle) runs on rank 0 alone.
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


def _rank_main(rank, world, port, local_ms, out_dir):
    # runs in a spawned process: one gloo rank
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms[rank], dist)
        value = bench.job_throughput(800, world, 10, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo(tmp_path):
    import torch.multiprocessing as mp

    world, port = 2, _free_port()
    local_ms = [30.0, 50.0]
    mp.start_processes(_rank_main, args=(world, port, local_ms, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        # the slowest rank's time, and both replicas' tokens over it
        assert g["ms"] == 50.0
        assert g["value"] == pytest.approx(800 * 2 * 10 / 0.050)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_throughput(25600, 1, 1000, 125.0) == pytest.approx(25600 * 1000 / 0.125)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0(oracle):
    # two CPU ranks: rank 0 times the oracle on its bounded sample, rank 1 exits 0
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0

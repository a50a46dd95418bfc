"""Host logic of the multi-replica benchmark, on CPU with gloo (world size 2).

With N > 1 every rank runs an independent replica of the layer on its own
GPU; the only cross-rank steps are the barrier around the timed region and
the MAX all-reduce of the elapsed time.  These tests run that host logic in
two gloo processes, and the reference arm under torchrun, where rank 0 alone
prints one line.
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

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, out_dir, rank_ms):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(rank_ms[rank], w, "cpu")
        val = bench.job_tokens_per_s(w, 4096, 100, ms)
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": val}, f)


def test_max_over_ranks_and_job_value_gloo(tmp_path):
    world = 2
    rank_ms = [12.5, 20.0]
    mp.spawn(_replica, args=(world, _free_port(), str(tmp_path), rank_ms), nprocs=world,
             join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    # every rank sees the slowest rank's time, and the whole-job value
    # counts the tokens of both replicas over that time
    for r in res:
        assert r["ms"] == max(rank_ms)
        assert r["value"] == pytest.approx(world * 4096 * 100 / (max(rank_ms) / 1e3), rel=1e-12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(7.0, 1, "cpu") == 7.0
    assert bench.job_tokens_per_s(1, 4096, 10, 100.0) == pytest.approx(409600.0)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched with two ranks: rank 0 times the
    oracle and prints one JSON line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny"

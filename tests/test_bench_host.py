"""Host logic of the benchmark's multi-rank mode, on CPU with gloo: each rank
runs its own replica, the line reports the sum of the ranks' bytes over the
slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    dev = torch.device("cpu")
    region_ms = [10.0, 12.5][rank]
    step_bytes = [1000.0, 1000.0][rank]
    out[rank] = (bench.reduce_max(region_ms, world, dev), bench.reduce_sum(step_bytes, world, dev),
                 bench.dist_env())
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
        got = dict(out)
    for rank in range(world):
        mx, total, env = got[rank]
        assert mx == 12.5          # slowest rank's time
        assert total == 2000.0     # all ranks' bytes
        assert env == (rank, world, rank)


def test_single_rank_reductions_are_identity():
    assert bench.reduce_max(3.0, 1, None) == 3.0
    assert bench.reduce_sum(4.0, 1, None) == 4.0


def test_reference_arm_under_two_ranks_prints_one_line():
    """torchrun with two CPU ranks: rank 0 times the oracle and prints one
    JSON line with the arm's fields, rank 1 exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "1", "--ref-budget-s", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == bench.STEP_CONFIG["workload"]

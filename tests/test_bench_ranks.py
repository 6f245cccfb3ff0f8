"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each with its
own timing, agree on the slowest rank's time (barrier + all-reduce MAX), which
sets the aggregate throughput; the reference arm prints only on rank 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch
    dist_mod = bench.init_dist(world, "gloo")
    bench.barrier(dist_mod)
    local_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
    agg = bench.max_over_ranks(local_ms, dist_mod, torch.device("cpu"))
    q.put((rank, agg))
    dist_mod.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 20.0, 1: 20.0}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None, None) == 3.5


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_launch_stats_window_means():
    """Windowed means of consecutive launches: exact on a known sequence,
    absent when there are fewer launches than one window."""
    sys.path.insert(0, ROOT)
    import bench
    per = [1.0] * 20 + [3.0] * 20
    st = bench.launch_stats(per)
    assert st["median"] == 2.0 and st["min"] == 1.0 and st["max"] == 3.0 and st["launches"] == 40
    assert st["window_mean_20"] == {"min": 1.0, "max": 3.0}
    st = bench.launch_stats([2.0, 4.0, 6.0, 8.0], window=2)
    assert st["window_mean_2"] == {"min": 3.0, "max": 7.0}
    assert "window_mean_20" not in bench.launch_stats([1.0] * 19)

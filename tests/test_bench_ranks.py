"""The benchmark's host logic on CPU: it refuses to run on more than one GPU
(the library is single-GPU code), the reference arm prints only on rank 0 of
a multi-rank launch, both arms describe the same workload, and the per-launch
statistics are right on known sequences."""
import json
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_more_than_one_gpu_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 2
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["unavailable"].startswith("one GPU only")
    assert line["n_gpus"] == 2


def test_multi_rank_launch_is_refused_on_every_rank():
    for rank in ("0", "1"):
        env = dict(os.environ, RANK=rank, WORLD_SIZE="2", LOCAL_RANK=rank)
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")], env=env,
                           capture_output=True, text=True, timeout=120)
        assert r.returncode == 2
        assert ("one GPU only" in r.stdout) == (rank == "0")


def test_bench_has_no_collective():
    with open(os.path.join(ROOT, "bench.py")) as f:
        src = f.read()
    assert not re.search(r"init_process_group|nccl|all_reduce", src)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_matches_our_config(monkeypatch, capsys):
    """The oracle arm prints the benchmark's metric, unit and config, on a
    tiny row sample (the oracle's row timing is stubbed to keep this quick)."""
    bench = _bench()
    import oracle
    calls = []

    def fake_gemm(A, B, dtype="bf16", rows=None):
        calls.append(rows)
        return None, None
    monkeypatch.setattr(oracle, "gemm", fake_gemm)
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["config"] == bench.CONFIG and line["unit"] == "TFLOP/s" and line["higher_is_better"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert len(calls) == 1 + 3 + 2  # the timing probe, the warm-up and the timed steps


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_launch_stats_window_means():
    """Windowed means of consecutive launches: exact on a known sequence,
    absent when there are fewer launches than one window."""
    bench = _bench()
    per = [1.0] * 20 + [3.0] * 20
    st = bench.launch_stats(per)
    assert st["median"] == 2.0 and st["min"] == 1.0 and st["max"] == 3.0 and st["launches"] == 40
    assert st["window_mean_20"] == {"min": 1.0, "max": 3.0}
    st = bench.launch_stats([2.0, 4.0, 6.0, 8.0], window=2)
    assert st["window_mean_2"] == {"min": 3.0, "max": 7.0}
    assert "window_mean_20" not in bench.launch_stats([1.0] * 19)


def test_oracle_rate_restores_thread_count():
    """The one-core CPU baseline leaves the oracle on all its threads."""
    bench = _bench()
    import oracle
    from blackwell_tensor_core_gb300 import workloads as wl
    before = oracle.num_threads()
    g = wl.generator(5)
    A = wl.bits(wl.normal_matrix(8, 64, 1.0, g))
    B = wl.bits(wl.normal_matrix(64, 32, 1.0, g))
    r = bench.oracle_rate(A, B, 0.01, threads=1)
    assert r["cores"] == 1 and r["kind"] == "oracle" and r["value"] > 0
    assert oracle.num_threads() == before

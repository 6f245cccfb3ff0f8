"""Failure detection without a GPU fault: the stage barriers are made to wait
for bytes that never arrive (an inflated transaction count), every bounded
wait gives up after a short limit, the kernel unwinds and frees its TMEM, and
the host reads BWG_ERR_TIMEOUT from the device error word.  The context must
stay usable: a normal call afterwards gives the right answer."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl
from gpu_util import gpu_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


@pytest.mark.parametrize("kind,M,sched", [("2cta", 256, "static"), ("1cta", 256, "static"),
                                          ("2cta_mc", 512, "static"), ("2cta_2c", 512, "static"),
                                          ("2cta_2c", 512, "clc"), (None, 64, "static")])
def test_stalled_stage_barrier_times_out_and_context_survives(kind, M, sched, monkeypatch):
    from blackwell_tensor_core_gb300 import ops
    from gpu_util import forced_kernel
    monkeypatch.setenv("BWG_SCHED", sched)
    g = wl.generator(7000)
    A = wl.randint_matrix(M, 256, -2, 2, g)
    B = wl.randint_matrix(256, 256, -2, 2, g)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros((M, 256), dtype=torch.float32, device="cuda")
    ops.set_watchdog_ns(50_000_000)  # 50 ms
    ops.debug_set_tx_extra(1024)
    try:
        with forced_kernel(kind):
            ops.gemm_bf16(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, 256, 256, 256, 256, 256,
                          wl.OUT_FP32, torch.cuda.current_stream().cuda_stream)
        st, word = ops.last_device_error()
    finally:
        ops.debug_set_tx_extra(0)
        ops.set_watchdog_ns(0)
    assert st == 5, "expected BWG_ERR_TIMEOUT, got %d (%#x)" % (st, word)
    assert (word >> 56) == 1
    # the context still works and gives the exact answer
    Dg, _ = gpu_gemm(A, B, wl.OUT_FP32, kind)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    assert np.array_equal(Dg.double().numpy(), Dref)


@pytest.mark.parametrize("mode,K", [("split", 256), ("whole", 256), ("streamk", 4864)])
def test_small_m_modes_time_out_and_context_survives(mode, K, monkeypatch):
    """The small-M kernel in each of its work splits -- cluster split (CTAs
    of a cluster also wait for each other's partials), whole tiles, and
    stream-K -- gives up on a stage barrier that cannot complete, reports
    BWG_ERR_TIMEOUT, and the next call is exact."""
    from blackwell_tensor_core_gb300 import ops
    M, N = 64, 256
    if mode == "whole":
        monkeypatch.setenv("BWG_SMALL_M_SPLIT", "0")
    if mode == "streamk":
        monkeypatch.setenv("BWG_STREAMK", "1")
    pl = ops.plan(M, N, K)
    assert (pl.split > 1) == (mode == "split") and (pl.streamk == 1) == (mode == "streamk")
    g = wl.generator(7050 + K)
    A = wl.randint_matrix(M, K, -2, 2, g)
    B = wl.randint_matrix(K, N, -2, 2, g)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    ops.set_watchdog_ns(50_000_000)  # 50 ms
    ops.debug_set_tx_extra(1024)
    try:
        ops.gemm_bf16(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K, N, N, wl.OUT_FP32,
                      torch.cuda.current_stream().cuda_stream)
        st, word = ops.last_device_error()
    finally:
        ops.debug_set_tx_extra(0)
        ops.set_watchdog_ns(0)
    assert st == 5 and (word >> 56) == 1, (st, hex(word))
    Dg, _ = gpu_gemm(A, B, wl.OUT_FP32, None)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    assert np.array_equal(Dg.double().numpy(), Dref)


@pytest.mark.parametrize("sched", ["clc", "static"])
def test_grouped_stalled_stage_barrier_times_out(sched, monkeypatch):
    """The grouped two-consumer kernel (dynamic and static scheduling) gives
    up on a stage barrier that cannot complete, reports BWG_ERR_TIMEOUT, and
    the next call is exact."""
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_SCHED", sched)
    counts = [300, 700]
    off = wl.offsets_from_counts(counts)
    g = wl.generator(7100)
    A = wl.randint_matrix(int(off[-1]), 128, -2, 2, g)
    Bs = [wl.randint_matrix(128, 256, -2, 2, g) for _ in counts]
    dev = torch.device("cuda")
    Ad, Bd, offd = A.to(dev), [b.to(dev) for b in Bs], torch.from_numpy(off).to(dev)
    D = torch.zeros((A.shape[0], 256), dtype=torch.bfloat16, device=dev)
    ops.set_watchdog_ns(50_000_000)
    ops.debug_set_tx_extra(1024)
    try:
        ops.grouped_gemm(Ad, Bd, offd, out=D)
        st, word = ops.last_device_error()
    finally:
        ops.debug_set_tx_extra(0)
        ops.set_watchdog_ns(0)
    assert st == 5 and (word >> 56) == 1, (st, hex(word))
    ops.grouped_gemm(Ad, Bd, offd, out=D)
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    Dref, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off)
    assert np.array_equal(wl.bits(D.cpu()), oracle.round_to(Dref, "bf16"))

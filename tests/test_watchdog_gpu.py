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


@pytest.mark.parametrize("kind,M", [("2cta", 256), ("1cta", 256), ("2cta_mc", 512), ("2cta_2c", 512),
                                    (None, 64)])
def test_stalled_stage_barrier_times_out_and_context_survives(kind, M):
    from blackwell_tensor_core_gb300 import ops
    from gpu_util import forced_kernel
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

"""GPU parity of how the small-M kernel fills its stage ring: one load of
B^T per stage through the 3-D channel-group view, and two stages per load
of B^T and of A.  Every work split (whole tiles, cluster split with odd
slices, stream-K) and an odd ring are exact on integer inputs and give the
same bits as one-stage loads (BWG_SMALL_M_PAIRS=0)."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl
from gpu_util import assert_bits_equal, gpu_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


# (M, N, K, env, expected (split > 1, streamk, bt_loads, pair_loads))
CASES = [
    ((72, 16384, 512), {}, (False, 0, 1, 1)),                       # whole tiles
    ((72, 4096, 2048), {}, (True, 0, 1, 1)),                        # cluster split
    ((40, 2048, 832), {"BWG_SMALL_M_SPLIT": "4"}, (True, 0, 1, 1)),  # 13 k-blocks: odd slices
    ((72, 4096, 4864), {"BWG_STREAMK": "1"}, (False, 1, 1, 1)),     # stream-K segments
    ((128, 4096, 640), {}, (True, 0, 1, 1)),                        # 7-stage ring
    ((72, 1000, 512), {}, (True, 0, 2, 0)),                         # N % 64 != 0: two boxes
    ((72, 16384, 1000), {}, (False, 0, 1, 0)),                      # K % 64 != 0: single stages
]


@pytest.mark.parametrize("shape,env,want", CASES)
def test_ring_fill_exact_and_same_bits_as_single_stage_loads(shape, env, want, monkeypatch):
    from blackwell_tensor_core_gb300 import ops
    M, N, K = shape
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    pl = ops.plan(M, N, K, wl.OUT_FP32)
    assert (pl.split > 1, pl.streamk, pl.bt_loads, pl.pair_loads) == want, shape
    g = wl.generator(9500 + M + N + K)
    A = wl.randint_matrix(M, K, -2, 2, g)
    B = wl.randint_matrix(K, N, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D, _ = gpu_gemm(A, B, wl.OUT_FP32)
    assert np.array_equal(D.double().numpy(), Dref), shape
    D16, _ = gpu_gemm(A, B, wl.OUT_BF16)
    assert_bits_equal(D16, oracle.round_to(Dref, "bf16"), "bf16 %s" % (shape,))
    # random inputs: bit-identical with and without two-stage loads
    A = wl.normal_matrix(M, K, 1.0, g)
    B = wl.normal_matrix(K, N, 1.0, g)
    D1, _ = gpu_gemm(A, B, wl.OUT_BF16)
    monkeypatch.setenv("BWG_SMALL_M_PAIRS", "0")
    assert ops.plan(M, N, K).pair_loads == 0
    D0, _ = gpu_gemm(A, B, wl.OUT_BF16)
    assert torch.equal(D0, D1), shape


@pytest.mark.parametrize("shape", [(72, 16384, 512), (16, 4096, 2048), (72, 1024, 832)])
def test_b_stored_nk_ring_fill_exact(shape, monkeypatch):
    """B stored [N, K]: one 128-row box a stage, two stages per load when K is
    a multiple of 64; exact, and the same bits without two-stage loads."""
    from blackwell_tensor_core_gb300 import ops
    M, N, K = shape
    g = wl.generator(9600 + K)
    A = wl.randint_matrix(M, K, -2, 2, g)
    Bt = wl.randint_matrix(N, K, -2, 2, g)
    dev = torch.device("cuda")
    Ad, Bd = A.to(dev), Bt.to(dev)
    h = torch.cuda.current_stream().cuda_stream

    def run():
        D = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        ops.gemm_bf16_nt(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K, K, N, wl.OUT_FP32, h)
        torch.cuda.synchronize()
        st, word = ops.last_device_error()
        assert st == 0, hex(word)
        return D.cpu()

    D1 = run()
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(Bt.t().contiguous()))
    assert np.array_equal(D1.double().numpy(), Dref), shape
    monkeypatch.setenv("BWG_SMALL_M_PAIRS", "0")
    assert torch.equal(run(), D1)

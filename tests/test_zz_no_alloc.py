"""The no-allocation small-M entry point, checked against gemm_bf16.

gemm_bf16_small_m_noalloc is for callers that cannot let the library call
cudaMalloc (all device memory handed to the caller's own pool allocator, or a
loop that must never stall on the allocator): it keeps the stream-K
kernel's partial sums in a fixed device array of the library.  This file runs
last so that, should it fail, every other test has already run; it also
passes on its own in a fresh process.  Each case makes two calls in a row on
the shared array and compares both with gemm_bf16, within the library's
tolerance |D - D_ref| <= 2^-7 |D_ref| + 1e-3 sum_k |a_ik b_kj|."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

OUT = {wl.OUT_BF16: torch.bfloat16, wl.OUT_FP32: torch.float32, wl.OUT_FP16: torch.float16}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    path = build.build()
    L = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    for name in ("gemm_bf16", "gemm_bf16_small_m_noalloc"):
        f = getattr(L, name)
        f.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp]
        f.restype = i
    return L


def _call(fn, A, B, D, M, N, K, out):
    st = fn(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, K, N, N, out,
            torch.cuda.current_stream().cuda_stream)
    assert st == 0, "status %d" % st


@pytest.mark.parametrize("M,N,K,out", [(72, 16384, 7168, wl.OUT_BF16), (16, 1000, 4096, wl.OUT_FP32),
                                       (128, 4104, 640, wl.OUT_BF16), (40, 256, 10240, wl.OUT_FP16)])
def test_noalloc_matches_gemm_bf16_on_two_calls(lib, M, N, K, out):
    g = wl.generator(8000 + M + N)
    A = wl.normal_matrix(M, K, 1.0, g)
    B = wl.normal_matrix(K, N, 1.0, g)
    Ad, Bd = A.cuda(), B.cuda()
    D_ref = torch.empty((M, N), dtype=OUT[out], device="cuda")
    _call(lib.gemm_bf16, Ad, Bd, D_ref, M, N, K, out)
    # S (the absolute-product sums) on sampled outputs sets the tolerance
    rng = np.random.default_rng(M + N)
    I = rng.integers(0, M, 3000)
    J = rng.integers(0, N, 3000)
    _, S = oracle.gemm_elements(wl.bits(A), wl.bits(B), I, J)
    want = D_ref.double().cpu().numpy()
    for _ in range(2):
        D = torch.full((M, N), float("nan"), dtype=OUT[out], device="cuda")
        _call(lib.gemm_bf16_small_m_noalloc, Ad, Bd, D, M, N, K, out)
        torch.cuda.synchronize()
        got = D.double().cpu().numpy()
        assert np.isfinite(got).all()
        err = np.abs(got[I, J] - want[I, J])
        assert (err <= 2.0 ** -7 * np.abs(want[I, J]) + 1e-3 * S).all()


def test_noalloc_integer_inputs_equal_exactly(lib):
    g = wl.generator(8100)
    A = wl.randint_matrix(72, 3000, -1, 1, g)
    B = wl.randint_matrix(3000, 2048, -1, 1, g)
    Ad, Bd = A.cuda(), B.cuda()
    D_ref = torch.empty((72, 2048), dtype=torch.float32, device="cuda")
    _call(lib.gemm_bf16, Ad, Bd, D_ref, 72, 2048, 3000, wl.OUT_FP32)
    for _ in range(2):
        D = torch.empty_like(D_ref)
        _call(lib.gemm_bf16_small_m_noalloc, Ad, Bd, D, 72, 2048, 3000, wl.OUT_FP32)
        torch.cuda.synchronize()
        assert torch.equal(D, D_ref)


def test_noalloc_rejects_sizes_beyond_its_buffer(lib):
    # 128 rows x 262144 columns: 2048 tiles of partial sums do not fit in 32 MiB
    M, N, K = 128, 262144, 1024
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = lib.gemm_bf16_small_m_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, K, N, N,
                                       wl.OUT_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == 6  # BWG_ERR_SCRATCH_LIMIT
    st = lib.gemm_bf16_small_m_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), 129, 256, K, K, 256,
                                       256, wl.OUT_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == 3  # more than 128 rows: not the small-M kernel

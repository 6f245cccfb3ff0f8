"""The no-allocation small-M entry point, checked against the oracle and
against gemm_bf16.

gemm_bf16_small_m_noalloc is for callers that cannot let the library call
cudaMalloc: a process that has handed all device memory to its own pool
allocator (a library allocation would fail, or eat into the pool's budget),
or a loop that must never stall on the allocator.  It keeps the stream-K
kernel's partial sums in a fixed device array of the library.  This file runs
last so that, should it fail, every other test has already run; it also
passes on its own in a fresh process.  Each case makes two calls in a row on
the shared array and compares both, element by element, with the CPU oracle
and with gemm_bf16's output, within the library's tolerance
|D - D_ref| <= 2^-7 |D_ref| + 1e-3 sum_k |a_ik b_kj|."""
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
def test_noalloc_matches_oracle_and_gemm_bf16_on_two_calls(lib, M, N, K, out):
    g = wl.generator(8000 + M + N)
    A = wl.normal_matrix(M, K, 1.0, g)
    B = wl.normal_matrix(K, N, 1.0, g)
    Ad, Bd = A.cuda(), B.cuda()
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B))
    D_lib = torch.empty((M, N), dtype=OUT[out], device="cuda")
    _call(lib.gemm_bf16, Ad, Bd, D_lib, M, N, K, out)
    torch.cuda.synchronize()
    lib_vals = D_lib.double().cpu().numpy()
    assert not oracle.bound_violations(lib_vals, Dref, S).any()
    for call in range(2):
        D = torch.full((M, N), float("nan"), dtype=OUT[out], device="cuda")
        _call(lib.gemm_bf16_small_m_noalloc, Ad, Bd, D, M, N, K, out)
        torch.cuda.synchronize()
        got = D.double().cpu().numpy()
        bad = oracle.bound_violations(got, Dref, S)
        assert not bad.any(), "call %d: %d outputs outside the bound around the oracle" % (call, bad.sum())
        bad = oracle.bound_violations(got, lib_vals, S)
        assert not bad.any(), "call %d: %d outputs outside the bound around gemm_bf16" % (call, bad.sum())


def test_noalloc_integer_inputs_equal_exactly(lib):
    """Integer inputs: every partial sum is exact in FP32, so both calls equal
    the oracle (and gemm_bf16) bit for bit, however the k-blocks are shared."""
    g = wl.generator(8100)
    A = wl.randint_matrix(72, 3000, -1, 1, g)
    B = wl.randint_matrix(3000, 2048, -1, 1, g)
    Ad, Bd = A.cuda(), B.cuda()
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D_lib = torch.empty((72, 2048), dtype=torch.float32, device="cuda")
    _call(lib.gemm_bf16, Ad, Bd, D_lib, 72, 2048, 3000, wl.OUT_FP32)
    for _ in range(2):
        D = torch.empty_like(D_lib)
        _call(lib.gemm_bf16_small_m_noalloc, Ad, Bd, D, 72, 2048, 3000, wl.OUT_FP32)
        torch.cuda.synchronize()
        assert np.array_equal(D.cpu().double().numpy(), Dref)
        assert torch.equal(D, D_lib)


def test_noalloc_ignores_the_tile_stride_override(lib, monkeypatch):
    """The planner's tile-stride override applies to gemm_bf16 only: the
    no-allocation kernel always stores 128-column tiles, so the override
    neither changes its result nor its scratch sizing."""
    monkeypatch.setenv("BWG_SMALL_M_TILE_N", "64")
    g = wl.generator(8200)
    A = wl.randint_matrix(72, 2048, -1, 1, g)
    B = wl.randint_matrix(2048, 4096, -1, 1, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D = torch.empty((72, 4096), dtype=torch.float32, device="cuda")
    _call(lib.gemm_bf16_small_m_noalloc, A.cuda(), B.cuda(), D, 72, 4096, 2048, wl.OUT_FP32)
    torch.cuda.synchronize()
    assert np.array_equal(D.cpu().double().numpy(), Dref)


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

"""GPU parity of the B-stored-as-[N, K] entry points (gemm_*_nt and
grouped_gemm_*_nt): D = A x B^T, B entering the tensor cores as a K-major
operand.  The oracle multiplies A by the transpose of the stored B."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl
from gpu_util import OUT_TORCH, assert_bits_equal, assert_within_bound, forced_kernel, in_dtype_name

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


def gemm_nt(A, Bt, out_dtype, kind=None, ldb=None, ldd=None, sentinel=float("nan")):
    """A [M, K] and Bt [N, K] on the CPU; returns D [M, N] and the full D buffer (CPU)."""
    from blackwell_tensor_core_gb300 import ops
    M, K = A.shape
    N = Bt.shape[0]
    ldb = ldb or K
    ldd = ldd or N
    Bbuf = torch.zeros((N, ldb), dtype=Bt.dtype)
    Bbuf[:, :K] = Bt
    dev = torch.device("cuda")
    Ad, Bd = A.to(dev), Bbuf.to(dev)
    D = torch.full((M, ldd), sentinel, dtype=OUT_TORCH[out_dtype], device=dev)
    fn = ops.gemm_bf16_nt if A.dtype == torch.bfloat16 else ops.gemm_fp16_nt
    with forced_kernel(kind):
        fn(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K, ldb, ldd, out_dtype,
           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    full = D.cpu()
    return full[:, :N], full


def ref_nt(A, Bt):
    """Oracle product of A and the transpose of the stored B."""
    return oracle.gemm(wl.bits(A), wl.bits(Bt.t().contiguous()), dtype=in_dtype_name(A))


@pytest.mark.parametrize("kind,M,N,K", [("2cta_2c", 1000, 1000, 520), ("2cta", 600, 704, 304),
                                        ("1cta", 300, 520, 200), ("2cta_mc", 1100, 600, 256),
                                        (None, 72, 16384, 512), (None, 72, 4096, 1024),
                                        (None, 100, 1000, 640)])
def test_nt_integer_exact_every_kernel(kind, M, N, K):
    """Exact on integer inputs with every kernel kind (the small-M shapes run
    whole tiles, the cluster split and a ragged last tile), FP32 and BF16 out."""
    g = wl.generator(9100 + M + N)
    A = wl.randint_matrix(M, K, -2, 2, g)
    Bt = wl.randint_matrix(N, K, -2, 2, g)
    Dref, _ = ref_nt(A, Bt)
    D, _ = gemm_nt(A, Bt, wl.OUT_FP32, kind)
    assert np.array_equal(D.double().numpy(), Dref), kind
    D16, _ = gemm_nt(A, Bt, wl.OUT_BF16, kind)
    assert_bits_equal(D16, oracle.round_to(Dref, "bf16"), "nt bf16 %s" % kind)


@pytest.mark.parametrize("shape", [(257, 391, 330), (72, 5000, 4096), (1, 128, 64), (600, 3000, 2048)])
def test_nt_random_within_bound_and_padded_ldb(shape):
    """Random inputs within the bound, FP16 too, with padded leading
    dimensions of B and D (D's padding untouched)."""
    M, N, K = shape
    if (K * 2) % 16 or (N * 2) % 16:
        K += (8 - K % 8) % 8
        N += (8 - N % 8) % 8
    g = wl.generator(9200 + M)
    A = wl.normal_matrix(M, K, 1.0, g)
    Bt = wl.normal_matrix(N, K, 1.0, g)
    Dref, S = ref_nt(A, Bt)
    D, full = gemm_nt(A, Bt, wl.OUT_BF16, None, ldb=K + 64, ldd=N + 16, sentinel=3.0)
    assert_within_bound(D, Dref, S, "nt random %s" % (shape,))
    assert (full[:, N:] == 3.0).all()
    Ah, Bh = A.to(torch.float16), Bt.to(torch.float16)
    Dh_ref, Sh = ref_nt(Ah, Bh)
    Dh, _ = gemm_nt(Ah, Bh, wl.OUT_FP16, None)
    assert_within_bound(Dh, Dh_ref, Sh, "nt fp16 %s" % (shape,))


def test_nt_large_8192_sampled():
    """The benchmark's shape with B stored [N, K]: 20,000 sampled outputs."""
    c = wl.large_case()
    Bt = c.B.t().contiguous()
    D, _ = gemm_nt(c.A, Bt, wl.OUT_BF16, None)
    rng = np.random.default_rng(77)
    I, J = rng.integers(0, c.M, 20000), rng.integers(0, c.N, 20000)
    ref, S = oracle.gemm_elements(wl.bits(c.A), wl.bits(c.B), I, J)
    got = D.double().numpy()[I, J]
    assert (np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-3 * S).all()


def test_nt_small_m_method_workload_full():
    c = wl.small_m_case()
    Bt = c.B.t().contiguous()
    D, _ = gemm_nt(c.A, Bt, wl.OUT_BF16, None)
    Dref, S = oracle.gemm(wl.bits(c.A), wl.bits(c.B))
    assert_within_bound(D, Dref, S, "nt small-M 72x16384x7168")


def test_nt_bad_leading_dimension():
    from blackwell_tensor_core_gb300 import ops
    A = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    Bt = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((16, 32), dtype=torch.bfloat16, device="cuda")
    h = torch.cuda.current_stream().cuda_stream
    st = ops.lib().gemm_bf16_nt(A.data_ptr(), Bt.data_ptr(), D.data_ptr(), 16, 32, 64, 64, 48, 32, 0, h)
    assert st == 1  # ldb < K
    st = ops.lib().gemm_bf16_nt(A.data_ptr(), Bt.data_ptr(), D.data_ptr(), 16, 32, 64, 64, 68, 32, 0, h)
    assert st == 2  # ldb * 2 not a multiple of 16 bytes


@pytest.mark.parametrize("swiglu,one_consumer,sched", [(False, False, "clc"), (True, False, "clc"),
                                                       (False, True, "static"), (True, True, "static"),
                                                       (False, False, "static")])
def test_grouped_nt_exact_and_matches_row_major(swiglu, one_consumer, sched, monkeypatch):
    """Grouped expert product with weights stored [N, K] (plain and SwiGLU,
    both grouped kernels and both schedulers, empty and ragged groups): exact
    on integer inputs, and the same results as the [K, N] entry point on the
    transposed weights."""
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_SCHED", sched)
    if one_consumer:
        monkeypatch.setenv("BWG_GROUPED_1C", "1")
    counts = [300, 0, 513, 7, 256]
    off = wl.offsets_from_counts(counts)
    g = wl.generator(9300 + int(swiglu))
    K, N = 320, 512
    A = wl.randint_matrix(int(off[-1]), K, -1, 1, g)
    Bts = [wl.randint_matrix(N, K, -1, 1, g) for _ in counts]
    dev = torch.device("cuda")
    Ad = A.to(dev)
    offd = torch.from_numpy(off).to(dev)
    D_nt = ops.grouped_gemm(Ad, [b.to(dev) for b in Bts], offd, swiglu=swiglu, b_transposed=True)
    D_nn = ops.grouped_gemm(Ad, [b.t().contiguous().to(dev) for b in Bts], offd, swiglu=swiglu)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    assert torch.equal(D_nt, D_nn)
    if not swiglu:
        Dref, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(b.t().contiguous()) for b in Bts], off)
        assert np.array_equal(wl.bits(D_nt.cpu()), oracle.round_to(Dref, "bf16"))

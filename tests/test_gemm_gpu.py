"""GPU parity of the dense kernels against the CPU oracle (through the C ABI).

Acceptance: bit-exact where the inputs are integers and every partial sum is
exact in binary32; otherwise |D - D_ref| <= 2^-7 |D_ref| + 1e-3 S elementwise
(S = sum_k |a_ik b_kj|), the bound the method states, for every output type."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl
from gpu_util import OUT_TORCH, assert_bits_equal, assert_within_bound, gpu_gemm, in_dtype_name

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


# ---------------------------------------------------------------- exact ----

@pytest.mark.parametrize("kind", ["2cta", "1cta", "2cta_mc"])
def test_tile_case_exact(kind):
    """256x256x512 integers in {-2..2}, FP32 out: every partial sum is an
    integer below 2^24, so the result is exact in any summation order."""
    c = wl.tile_case()
    D, _ = gpu_gemm(c.A, c.B, wl.OUT_FP32, kind)
    Dref, _ = oracle.gemm(wl.bits(c.A), wl.bits(c.B))
    assert np.array_equal(D.double().numpy(), Dref)


@pytest.mark.parametrize("kind", ["2cta", "1cta", "2cta_mc"])
@pytest.mark.parametrize("out", [wl.OUT_BF16, wl.OUT_FP16])
def test_integer_inputs_rounded_output_exact(kind, out):
    g = wl.generator(2001)
    A = wl.randint_matrix(384, 1024, -2, 2, g)
    B = wl.randint_matrix(1024, 520, -2, 2, g)
    D, _ = gpu_gemm(A, B, out, kind)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    assert_bits_equal(D, oracle.round_to(Dref, "fp16" if out == wl.OUT_FP16 else "bf16"), kind)


@pytest.mark.parametrize("M", [1, 16, 72, 100, 128])
def test_small_m_integer_exact(M):
    g = wl.generator(2002 + M)
    A = wl.randint_matrix(M, 640, -2, 2, g)
    B = wl.randint_matrix(640, 1000, -2, 2, g)
    D, _ = gpu_gemm(A, B, wl.OUT_FP32, None)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    assert np.array_equal(D.double().numpy(), Dref)
    D16, _ = gpu_gemm(A, B, wl.OUT_BF16, None)
    assert_bits_equal(D16, oracle.round_to(Dref, "bf16"), "small_m bf16")


# ------------------------------------------------------- bound, ragged -----

SHAPES = [(520, 600, 456), (300, 264, 72), (129, 8, 8), (256, 256, 64), (1000, 136, 1000),
          (257, 520, 40), (768, 1024, 2048)]


@pytest.mark.parametrize("kind", ["2cta", "1cta", "2cta_mc"])
@pytest.mark.parametrize("shape", SHAPES)
def test_random_shapes_within_bound(kind, shape):
    M, N, K = shape
    g = wl.generator(3000 + M + N + K)
    A = wl.normal_matrix(M, K, 1.0, g)
    B = wl.normal_matrix(K, N, 1.0, g)
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B))
    for out in (wl.OUT_BF16, wl.OUT_FP32):
        D, _ = gpu_gemm(A, B, out, kind)
        assert_within_bound(D, Dref, S, "%s %s out=%d" % (kind, shape, out))


@pytest.mark.parametrize("shape", [(1, 8, 8), (17, 200, 104), (72, 1000, 520), (128, 384, 64),
                                   (16, 16, 16), (33, 4104, 1000)])
@pytest.mark.parametrize("out", [wl.OUT_BF16, wl.OUT_FP32, wl.OUT_FP16])
def test_small_m_within_bound(shape, out):
    M, N, K = shape
    g = wl.generator(4000 + M + N + K)
    A = wl.normal_matrix(M, K, 1.0, g)
    B = wl.normal_matrix(K, N, 1.0, g)
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B))
    D, _ = gpu_gemm(A, B, out, None)
    assert_within_bound(D, Dref, S, "small_m %s out=%d" % (shape, out))


@pytest.mark.parametrize("kind", ["2cta", "1cta", "2cta_mc", None])
def test_fp16_inputs(kind):
    M = 72 if kind is None else 400
    g = wl.generator(5000)
    A = wl.normal_matrix(M, 328, 1.0, g, "fp16")
    B = wl.normal_matrix(328, 392, 1.0, g, "fp16")
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B), "fp16")
    for out in (wl.OUT_FP16, wl.OUT_FP32, wl.OUT_BF16):
        D, _ = gpu_gemm(A, B, out, kind)
        assert_within_bound(D, Dref, S, "fp16 in %s out=%d" % (kind, out))


@pytest.mark.parametrize("kind", ["2cta", "1cta", "2cta_mc", None])
def test_leading_dimensions_and_untouched_padding(kind):
    M = 90 if kind is None else 300
    N, K = 200, 136
    g = wl.generator(5100)
    A = wl.normal_matrix(M, K, 1.0, g)
    B = wl.normal_matrix(K, N, 1.0, g)
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B))
    D, full = gpu_gemm(A, B, wl.OUT_BF16, kind, lda=K + 24, ldb=N + 56, ldd=N + 40, sentinel=7.0)
    assert_within_bound(D, Dref, S, "strided %s" % kind)
    assert torch.all(full[:, N:] == 7.0), "padding columns of D were written"


def test_k_zero_writes_zeros_and_empty_is_noop():
    from blackwell_tensor_core_gb300 import ops
    D = torch.full((37, 64), 5.0, dtype=torch.bfloat16, device="cuda")
    ops.gemm_bf16(0, 0, D.data_ptr(), 37, 64, 0, 0, 0, 64, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.all(D == 0)
    ops.gemm_bf16(0, 0, 0, 0, 64, 10, 0, 0, 0, 0, torch.cuda.current_stream().cuda_stream)


def test_short_k_below_one_block():
    for K in (8, 16, 24, 56):
        g = wl.generator(5200 + K)
        A = wl.randint_matrix(300, K, -2, 2, g)
        B = wl.randint_matrix(K, 264, -2, 2, g)
        D, _ = gpu_gemm(A, B, wl.OUT_FP32, None)
        Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
        assert np.array_equal(D.double().numpy(), Dref)


def test_bad_arguments_return_status():
    from blackwell_tensor_core_gb300 import ops
    D = torch.empty((64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.BwgError) as e:
        ops.gemm_bf16(D.data_ptr() + 2, D.data_ptr(), D.data_ptr(), 64, 64, 64, 64, 64, 64, 0, 0)
    assert e.value.status == 2


def test_multicast_kernel_reads_only_this_gpus_memory():
    """The multicast kernel (two CTA pairs receiving each B box) may read only
    device memory of the GPU it runs on: operands in pinned host memory are
    refused with BWG_ERR_INVALID_ARG before any descriptor or launch, and the
    output is left untouched; the same call on device operands runs."""
    from blackwell_tensor_core_gb300 import ops
    from gpu_util import forced_kernel
    g = wl.generator(2300)
    M, N, K = 512, 512, 256
    A = wl.randint_matrix(M, K, -2, 2, g)
    B = wl.randint_matrix(K, N, -2, 2, g)
    Ad, Bd = A.cuda(), B.cuda()
    Ah, Bh = A.pin_memory(), B.pin_memory()
    D = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    h = torch.cuda.current_stream().cuda_stream
    L = ops.lib()
    with forced_kernel("2cta_mc"):
        for a, b in ((Ad, Bh), (Ah, Bd), (Ah, Bh)):
            st = L.gemm_bf16(a.data_ptr(), b.data_ptr(), D.data_ptr(), M, N, K, K, N, N, wl.OUT_FP32, h)
            assert st == 1
        torch.cuda.synchronize()
        assert bool((D == 7.0).all())
        assert L.gemm_bf16(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K, N, N, wl.OUT_FP32, h) == 0
    torch.cuda.synchronize()
    assert ops.last_device_error()[0] == 0
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    assert np.array_equal(D.cpu().double().numpy(), Dref)


# ------------------------------------------- full-size method workloads ----

def _sample_indices(M, N, n, seed, tile_m=256, tile_n=256):
    rng = np.random.default_rng(seed)
    I = list(rng.integers(0, M, n))
    J = list(rng.integers(0, N, n))
    # tile corners and edges
    for m in sorted({0, 127, 128, 255, tile_m, 511, 512, M - 1, M // 2}):
        for nn in sorted({0, 63, 64, 127, 128, 255, tile_n, N - 1}):
            if m < M and nn < N:
                I.append(m)
                J.append(nn)
    return np.array(I), np.array(J)


def _check_sampled(A, B, D, n, seed, what):
    M, N = D.shape
    I, J = _sample_indices(M, N, n, seed)
    Dref, S = oracle.gemm_elements(wl.bits(A), wl.bits(B), I, J, in_dtype_name(A))
    assert_within_bound(D[I, J], Dref, S, what)
    return I, J


def test_square_4096_sampled():
    c = wl.square_case()
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    assert torch.isfinite(D.float()).all()
    _check_sampled(c.A, c.B, D, 20000, 11, c.name)


def test_large_8192_sampled_in_bench_configuration():
    c = wl.large_case()
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    assert torch.isfinite(D.float()).all()
    _check_sampled(c.A, c.B, D, 20000, 12, c.name)
    # whole rows and columns at tile seams
    for r in (0, 255, 256, 8191):
        Dref, S = oracle.gemm(wl.bits(c.A[r:r + 1]), wl.bits(c.B))
        assert_within_bound(D[r:r + 1], Dref, S, "row %d" % r)


def test_small_m_method_workload_full():
    c = wl.small_m_case()
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    Dref, S = oracle.gemm(wl.bits(c.A), wl.bits(c.B))
    assert_within_bound(D, Dref, S, c.name)


# FP16 inputs (FP16 output) on the method's dense workloads: the same draws
# rounded to FP16; the oracle decodes the FP16 patterns.
def test_fp16_square_4096_sampled():
    c = wl.square_case(dtype="fp16")
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    assert D.dtype == torch.float16 and torch.isfinite(D.float()).all()
    _check_sampled(c.A, c.B, D, 20000, 21, c.name)


def test_fp16_large_8192_sampled():
    c = wl.large_case(dtype="fp16")
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    assert torch.isfinite(D.float()).all()
    _check_sampled(c.A, c.B, D, 20000, 22, c.name)
    for r in (0, 511, 512, 8191):
        Dref, S = oracle.gemm(wl.bits(c.A[r:r + 1]), wl.bits(c.B), "fp16")
        assert_within_bound(D[r:r + 1], Dref, S, "fp16 row %d" % r)


def test_fp16_small_m_method_workload_full():
    c = wl.small_m_case(dtype="fp16")
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    Dref, S = oracle.gemm(wl.bits(c.A), wl.bits(c.B), "fp16")
    assert_within_bound(D, Dref, S, c.name)


@pytest.mark.parametrize("kind", ["2cta", "1cta", "2cta_2c", "small_m"])
def test_fp16_integer_exact_every_kernel(kind):
    """Integer FP16 inputs: exact on every kernel kind, FP32 and FP16 output."""
    g = wl.generator(5500)
    M = 72 if kind == "small_m" else 600
    A = wl.randint_matrix(M, 320, -2, 2, g, "fp16")
    B = wl.randint_matrix(320, 520, -2, 2, g, "fp16")
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B), "fp16")
    D32, _ = gpu_gemm(A, B, wl.OUT_FP32, kind)
    assert np.array_equal(D32.double().numpy(), Dref)
    D16, _ = gpu_gemm(A, B, wl.OUT_FP16, kind)
    assert_bits_equal(D16, oracle.round_to(Dref, "fp16"), "fp16 out " + kind)


@pytest.mark.parametrize("kind", ["2cta", "1cta", "2cta_mc"])
def test_last_wave_split_matches_unsplit(kind, monkeypatch):
    """Half-width last-wave units (dynamic MMA N) give the same exact result
    as whole tiles; 2304 tiles of 128 or 256 rows leave a remainder that is
    split on both kernels."""
    g = wl.generator(5300)
    A = wl.randint_matrix(640, 512, -2, 2, g)
    B = wl.randint_matrix(512, 2304, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D1, _ = gpu_gemm(A, B, wl.OUT_FP32, kind)
    assert np.array_equal(D1.double().numpy(), Dref)
    monkeypatch.setenv("BWG_NO_TAIL_SPLIT", "1")
    D2, _ = gpu_gemm(A, B, wl.OUT_FP32, kind)
    assert np.array_equal(D2.double().numpy(), Dref)


@pytest.mark.parametrize("kind", ["2cta", "1cta", "2cta_mc"])
@pytest.mark.parametrize("out", [wl.OUT_FP32, wl.OUT_BF16])
def test_register_store_epilogue(kind, out, monkeypatch):
    """The epilogue that stores rows straight from registers (seven-stage
    ring) gives the same results, including ragged M and N edges."""
    monkeypatch.setenv("BWG_EPILOGUE", "direct")
    g = wl.generator(5400)
    A = wl.randint_matrix(520, 640, -2, 2, g)
    B = wl.randint_matrix(640, 600, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D, full = gpu_gemm(A, B, out, kind, ldd=608, sentinel=9.0)
    if out == wl.OUT_FP32:
        assert np.array_equal(D.double().numpy(), Dref)
    else:
        assert_bits_equal(D, oracle.round_to(Dref, "bf16"), "direct bf16")
    assert torch.all(full[:, 600:] == 9.0)


def test_multicast_kernel_at_8192_sampled():
    """The two-pair multicast kernel on the 8192^3 workload (odd and even
    unit rows, last-wave split) on sampled outputs and seam rows."""
    c = wl.large_case()
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype, "2cta_mc")
    _check_sampled(c.A, c.B, D, 8000, 14, c.name + " multicast")
    for r in (255, 256, 511, 512):
        Dref, S = oracle.gemm(wl.bits(c.A[r:r + 1]), wl.bits(c.B))
        assert_within_bound(D[r:r + 1], Dref, S, "row %d" % r)


# --------------------------------------------------- small-M stream-K ------

@pytest.mark.parametrize("shape", [(72, 1000, 4096), (16, 128, 8192), (128, 4104, 640), (72, 16384, 512)])
def test_small_m_streamk_exact_and_repeatable(shape, monkeypatch):
    """Stream-K shares each tile's k-blocks among several CTAs (up to ~20
    here); with integer inputs every partial sum is exact, so the result must
    equal the oracle bit for bit, on every repeat (the per-tile counters reset
    themselves) and with stream-K switched off."""
    M, N, K = shape
    g = wl.generator(5500 + M + N)
    A = wl.randint_matrix(M, K, -1, 1, g)
    B = wl.randint_matrix(K, N, -1, 1, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    for _ in range(3):
        D, _ = gpu_gemm(A, B, wl.OUT_FP32, None)
        assert np.array_equal(D.double().numpy(), Dref)
    monkeypatch.setenv("BWG_STREAMK", "0")
    D, _ = gpu_gemm(A, B, wl.OUT_FP32, None)
    assert np.array_equal(D.double().numpy(), Dref)
    monkeypatch.setenv("BWG_STREAMK", "1")
    D, _ = gpu_gemm(A, B, wl.OUT_FP32, None)
    assert np.array_equal(D.double().numpy(), Dref)


def test_small_m_streamk_bf16_bound_and_growing_workspace(monkeypatch):
    monkeypatch.setenv("BWG_STREAMK", "1")
    for (M, N, K) in [(40, 256, 10240), (72, 6000, 2048), (100, 12000, 3000)]:
        g = wl.generator(5600 + N)
        A = wl.normal_matrix(M, K, 1.0, g)
        B = wl.normal_matrix(K, N, 1.0, g)
        Dref, S = oracle.gemm(wl.bits(A), wl.bits(B))
        D, _ = gpu_gemm(A, B, wl.OUT_BF16, None)
        assert_within_bound(D, Dref, S, "streamk %s" % ((M, N, K),))


@pytest.mark.parametrize("shape", [(72, 4096, 7168), (70, 1000, 4096), (3, 640, 2048), (128, 4104, 640),
                                   (16, 2048, 4136), (72, 7168, 2048), (33, 312, 1016)])
def test_small_m_cluster_split_exact(shape, monkeypatch):
    """Cluster split of K (partials summed through distributed shared memory):
    exact on integer inputs for every output type, with ragged M (rows not a
    multiple of the cluster, fewer rows than CTAs), ragged K and N, and the
    same bits on every repeat; equal to the unsplit and stream-K results."""
    from blackwell_tensor_core_gb300 import ops
    M, N, K = shape
    pl = ops.plan(M, N, K)
    assert pl.split > 1, (shape, pl.split)
    g = wl.generator(5750 + M + N)
    A = wl.randint_matrix(M, K, -2, 2, g)
    B = wl.randint_matrix(K, N, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    for _ in range(2):
        D, _ = gpu_gemm(A, B, wl.OUT_FP32, None)
        assert np.array_equal(D.double().numpy(), Dref)
    D16, _ = gpu_gemm(A, B, wl.OUT_BF16, None)
    assert_bits_equal(D16, oracle.round_to(Dref, "bf16"), "split bf16 %s" % (shape,))
    Ah, Bh = A.to(torch.float16), B.to(torch.float16)
    Dh, _ = gpu_gemm(Ah, Bh, wl.OUT_FP16, None)
    assert_bits_equal(Dh, oracle.round_to(Dref, "fp16"), "split fp16 %s" % (shape,))
    monkeypatch.setenv("BWG_SMALL_M_SPLIT", "0")
    D0, _ = gpu_gemm(A, B, wl.OUT_FP32, None)
    assert np.array_equal(D0.double().numpy(), Dref)


def test_small_m_cluster_split_random_bound_and_padding():
    """Random inputs within the bound, bit-identical run to run, and a padded
    leading dimension of D left untouched."""
    from blackwell_tensor_core_gb300 import ops
    M, N, K = 72, 4096, 7168
    assert ops.plan(M, N, K).split == 4
    g = wl.generator(5790)
    A = wl.normal_matrix(M, K, 0.02, g)
    B = wl.normal_matrix(K, N, 0.02, g)
    D1, full = gpu_gemm(A, B, wl.OUT_BF16, None, ldd=N + 64, sentinel=7.0)
    D2, _ = gpu_gemm(A, B, wl.OUT_BF16, None, ldd=N + 64, sentinel=7.0)
    assert torch.equal(D1, D2)
    assert (full[:, N:] == 7.0).all()
    Dref, S = oracle.gemm(wl.bits(A), wl.bits(B))
    assert_within_bound(D1, Dref, S, "split random")


def test_small_m_streamk_on_a_side_stream():
    from blackwell_tensor_core_gb300 import ops
    g = wl.generator(5700)
    A = wl.randint_matrix(72, 2048, -2, 2, g)
    B = wl.randint_matrix(2048, 3000, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    s = torch.cuda.Stream()
    Ad, Bd = A.cuda(), B.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        D = ops.gemm(Ad, Bd, out_dtype=torch.float32, stream=s)
    s.synchronize()
    assert np.array_equal(D.cpu().double().numpy(), Dref)


def test_small_m_streamk_per_thread_default_streams(monkeypatch):
    """Two host threads run stream-K small-M products at once on their
    per-thread default streams: one handle (cudaStreamPerThread), two
    streams.  Each stream has its own partial-sum workspace, so both results
    are exact, every time."""
    import threading
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_STREAMK", "1")
    per_thread = 2  # cudaStreamPerThread
    g = wl.generator(5750)
    cases = []
    for i in range(2):
        A = wl.randint_matrix(72, 4096, -2, 2, g)
        B = wl.randint_matrix(4096, 3000 + 128 * i, -2, 2, g)
        Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
        cases.append((A.cuda(), B.cuda(), Dref))
    assert ops.plan(72, 3000, 4096).streamk == 1
    results = [[], []]
    errors = []
    dev = torch.cuda.current_device()

    def run(i):
        try:
            torch.cuda.set_device(dev)
            Ad, Bd, _ = cases[i]
            M, K = Ad.shape
            N = Bd.shape[1]
            Ds = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(20)]
            torch.cuda.synchronize()
            for D in Ds:
                ops.gemm_bf16(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K, N, N, wl.OUT_FP32,
                              per_thread)
                results[i].append(D)
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert ops.last_device_error()[0] == 0
    for i in range(2):
        for D in results[i]:
            assert np.array_equal(D.cpu().double().numpy(), cases[i][2])


def test_small_m_streamk_workspace_growth_refused_during_capture(monkeypatch):
    """A stream-K call that would have to grow its stream's workspace while
    the stream is being captured returns BWG_ERR_UNSUPPORTED, enqueues
    nothing and leaves the capture valid; after an eager call of that shape
    on the stream the same call records, and the replay is exact."""
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_STREAMK", "1")
    g = wl.generator(5760)
    A = wl.randint_matrix(72, 4096, -2, 2, g).cuda()
    B = wl.randint_matrix(4096, 6000, -2, 2, g).cuda()
    D = torch.zeros((72, 6000), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    L = ops.lib()
    args = (A.data_ptr(), B.data_ptr(), D.data_ptr(), 72, 6000, 4096, 4096, 6000, 6000, wl.OUT_FP32)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        st = L.gemm_bf16(*args, s.cuda_stream)
        # a no-op kernel keeps the captured graph non-empty
        D.add_(0)
    assert st == 3
    torch.cuda.synchronize()
    # eager call on the same stream makes the workspace; capture now records it
    assert L.gemm_bf16(*args, s.cuda_stream) == 0
    s.synchronize()
    graph2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph2, stream=s):
        assert L.gemm_bf16(*args, s.cuda_stream) == 0
    D.zero_()
    graph2.replay()
    torch.cuda.synchronize()
    Dref, _ = oracle.gemm(wl.bits(A.cpu()), wl.bits(B.cpu()))
    assert np.array_equal(D.cpu().double().numpy(), Dref)


@pytest.mark.parametrize("tile_n", [64, 80, 112, 128])
@pytest.mark.parametrize("out", [wl.OUT_BF16, wl.OUT_FP32])
@pytest.mark.parametrize("N", [1000, 1024])
def test_small_m_tile_stride(tile_n, out, N, monkeypatch):
    """Tiles that store fewer columns than the 128 the MMA spans: every
    column written exactly once, ragged last tile clipped, padding untouched.
    With N = 1024 a stride of 64 or 128 loads B^T through the channel-group
    view (one box a stage, two stages a load) and 80 or 112 as two boxes."""
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_SMALL_M_TILE_N", str(tile_n))
    pl = ops.plan(72, N, 640, out)
    grouped = N % 64 == 0 and tile_n % 64 == 0
    assert (pl.bt_loads, pl.pair_loads) == ((1, 1) if grouped else (2, 0))
    g = wl.generator(5800 + tile_n + N)
    A = wl.randint_matrix(72, 640, -2, 2, g)
    B = wl.randint_matrix(640, N, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D, full = gpu_gemm(A, B, out, None, ldd=N + 16, sentinel=5.0)
    if out == wl.OUT_FP32:
        assert np.array_equal(D.double().numpy(), Dref)
    else:
        assert_bits_equal(D, oracle.round_to(Dref, "bf16"), "tile_n %d" % tile_n)
    assert torch.all(full[:, N:] == 5.0)


@pytest.mark.parametrize("shape", [(512, 256, 512), (520, 600, 456), (1000, 136, 1000), (1536, 2304, 640),
                                   (129, 264, 72)])
def test_two_consumer_kernel_exact(shape):
    """512x256 tiles on a pair with two MMA consumers sharing each B stage:
    exact on integer inputs, including ragged M (second consumer's rows
    partly or wholly outside), ragged N and K, and the last-wave split."""
    M, N, K = shape
    g = wl.generator(5900 + M + N)
    A = wl.randint_matrix(M, K, -2, 2, g)
    B = wl.randint_matrix(K, N, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D, _ = gpu_gemm(A, B, wl.OUT_FP32, "2cta_2c")
    assert np.array_equal(D.double().numpy(), Dref)
    D16, _ = gpu_gemm(A, B, wl.OUT_BF16, "2cta_2c")
    assert_bits_equal(D16, oracle.round_to(Dref, "bf16"), "two consumers bf16")


def test_two_consumer_kernel_at_8192_sampled():
    c = wl.large_case()
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype, "2cta_2c")
    _check_sampled(c.A, c.B, D, 8000, 15, c.name + " two consumers")
    for r in (255, 256, 511, 512):
        Dref, S = oracle.gemm(wl.bits(c.A[r:r + 1]), wl.bits(c.B))
        assert_within_bound(D[r:r + 1], Dref, S, "row %d" % r)


@pytest.mark.parametrize("shape", [(2048, 5120, 128), (1536, 6656, 64), (1024, 13568, 64), (1800, 5120, 72)])
def test_two_consumer_last_wave_quarters_exact(shape, monkeypatch):
    """Shapes whose last wave is cut into quarters (one row block and one
    column half per unit, one MMA consumer idle) or whose second consumer
    has no rows: exact on integers, and equal with the cut switched off."""
    M, N, K = shape
    g = wl.generator(6200 + M + N)
    A = wl.randint_matrix(M, K, -2, 2, g)
    B = wl.randint_matrix(K, N, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D, _ = gpu_gemm(A, B, wl.OUT_FP32, "2cta_2c")
    assert np.array_equal(D.double().numpy(), Dref)
    monkeypatch.setenv("BWG_NO_TAIL_SPLIT", "1")
    D2, _ = gpu_gemm(A, B, wl.OUT_FP32, "2cta_2c")
    assert np.array_equal(D2.double().numpy(), Dref)


# ------------------------------------ cluster-launch-control scheduling ----

@pytest.mark.parametrize("shape,no_split", [((4096, 4096, 64), "0"), ((2560, 4864, 128), "0"),
                                            ((2560, 4864, 128), "1"), ((300, 520, 200), "0")])
def test_dynamic_schedule_exact(shape, no_split, monkeypatch):
    """Units claimed at run time (one pair launched per unit, running pairs
    cancel pending ones and take their units): 128 units on 76 pairs, 95
    tiles whose last wave is cut in quarters (or not), and a one-unit case."""
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_SCHED", "clc")
    monkeypatch.setenv("BWG_NO_TAIL_SPLIT", no_split)
    M, N, K = shape
    g = wl.generator(5600 + M)
    A = wl.randint_matrix(M, K, -2, 2, g)
    B = wl.randint_matrix(K, N, -2, 2, g)
    pl = ops.plan(M, N, K, wl.OUT_FP32, force_kernel=ops.KERNEL_2CTA_2C)
    assert pl.dynamic == 1 and pl.grid == 2 * pl.units
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D, _ = gpu_gemm(A, B, wl.OUT_FP32, "2cta_2c")
    assert np.array_equal(D.double().numpy(), Dref)
    D16, _ = gpu_gemm(A, B, wl.OUT_BF16, "2cta_2c")
    assert_bits_equal(D16, oracle.round_to(Dref, "bf16"), "dynamic bf16 %s" % (shape,))


def test_dynamic_schedule_8192_sampled(monkeypatch):
    monkeypatch.setenv("BWG_SCHED", "clc")
    c = wl.large_case()
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype, "2cta_2c")
    _check_sampled(c.A, c.B, D, 8000, 16, c.name + " dynamic")
    for r in (511, 512, 8191):
        Dref, S = oracle.gemm(wl.bits(c.A[r:r + 1]), wl.bits(c.B))
        assert_within_bound(D[r:r + 1], Dref, S, "row %d" % r)


# ------------------------------------------------- host-buffer entry point --

def _host_call(A, B, out_dtype, dA=None, dB=None, dD=None):
    from blackwell_tensor_core_gb300 import ops
    M, K = A.shape
    N = B.shape[1]
    hA, hB = A.pin_memory(), B.pin_memory()
    hD = torch.full((M, N), float("nan"), dtype=OUT_TORCH[out_dtype]).pin_memory()
    dA = dA if dA is not None else torch.empty((M, K), dtype=A.dtype, device="cuda")
    dB = dB if dB is not None else torch.empty((K, N), dtype=B.dtype, device="cuda")
    dD = dD if dD is not None else torch.empty((M, N), dtype=OUT_TORCH[out_dtype], device="cuda")
    ops.gemm_bf16_host(hA, hB, hD, dA, dB, dD)
    return hD, (dA, dB, dD)


@pytest.mark.parametrize("M", [700, 3000, 9000])
def test_host_entry_point_pipelined_chunks_exact(M):
    """1, 2 and 6 row chunks (whole 512-row tiles, a ragged last chunk): the
    copies, products and copies back are ordered by events; exact result."""
    g = wl.generator(5700 + M)
    A = wl.randint_matrix(M, 192, -2, 2, g)
    B = wl.randint_matrix(192, 264, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    hD, _ = _host_call(A, B, wl.OUT_FP32)
    torch.cuda.current_stream().synchronize()
    assert np.array_equal(hD.double().numpy(), Dref)


def test_host_entry_point_back_to_back_calls_reuse_buffers():
    """Two calls on one stream with the same device buffers and different
    inputs: the second call's copies wait for the first call's products, and
    each host result is that call's own product."""
    g = wl.generator(5800)
    A1 = wl.randint_matrix(4096, 128, -2, 2, g)
    B1 = wl.randint_matrix(128, 1024, -2, 2, g)
    A2 = wl.randint_matrix(4096, 128, -2, 2, g)
    B2 = wl.randint_matrix(128, 1024, -2, 2, g)
    h1, bufs = _host_call(A1, B1, wl.OUT_BF16)
    h2, _ = _host_call(A2, B2, wl.OUT_BF16, *bufs)
    torch.cuda.current_stream().synchronize()
    for A, B, h in ((A1, B1, h1), (A2, B2, h2)):
        Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
        assert_bits_equal(h, oracle.round_to(Dref, "bf16"), "host call")


def test_host_entry_point_8192_sampled():
    """The end-to-end configuration the benchmark times (8192^3, BF16 out)."""
    c = wl.large_case()
    hD, _ = _host_call(c.A, c.B, c.out_dtype)
    torch.cuda.current_stream().synchronize()
    _check_sampled(c.A, c.B, hD, 8000, 17, c.name + " host entry")


# --------------------------------------------- stream-K last wave (dense) ---

@pytest.mark.parametrize("shape", [(2560, 4864, 512), (2560, 4864, 520), (1024, 1024, 4096),
                                   (600, 2048, 1024)])
def test_streamk_last_wave_exact_and_repeatable(shape, monkeypatch):
    """Two-consumer kernel with the last wave shared out by k-block: 95 tiles
    (19 stream-K tiles, 4 pairs each), a ragged last k-block, 8 tiles over 76
    pairs (about 10 sharers a tile), ragged M.  Exact on integer inputs,
    FP32 and BF16 output, and bit-identical run to run on random inputs
    (partials are summed in pair order)."""
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_STREAMK_DENSE", "1")
    M, N, K = shape
    pl = ops.plan(M, N, K, wl.OUT_FP32, force_kernel=ops.KERNEL_2CTA_2C)
    assert pl.streamk == 1 and pl.sk_tiles > 0
    g = wl.generator(5900 + K)
    A = wl.randint_matrix(M, K, -2, 2, g)
    B = wl.randint_matrix(K, N, -2, 2, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    D, _ = gpu_gemm(A, B, wl.OUT_FP32, "2cta_2c")
    assert np.array_equal(D.double().numpy(), Dref)
    D16, _ = gpu_gemm(A, B, wl.OUT_BF16, "2cta_2c")
    assert_bits_equal(D16, oracle.round_to(Dref, "bf16"), "stream-K bf16 %s" % (shape,))
    Ar = wl.normal_matrix(M, K, 1.0, g)
    Br = wl.normal_matrix(K, N, 1.0, g)
    R1, _ = gpu_gemm(Ar, Br, wl.OUT_FP32, "2cta_2c")
    R2, _ = gpu_gemm(Ar, Br, wl.OUT_FP32, "2cta_2c")
    assert torch.equal(R1, R2)
    Rref, S = oracle.gemm(wl.bits(Ar), wl.bits(Br))
    assert_within_bound(R1, Rref, S, "stream-K random %s" % (shape,))


def test_streamk_off_matches_on_at_4096(monkeypatch):
    """4096^3 (52 of 128 tiles shared out): stream-K and the plain last wave
    give results within the bound on sampled outputs."""
    from blackwell_tensor_core_gb300 import ops
    c = wl.square_case()
    D0, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    monkeypatch.setenv("BWG_STREAMK_DENSE", "1")
    assert ops.plan(4096, 4096, 4096).streamk == 1
    D1, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    _check_sampled(c.A, c.B, D1, 4000, 31, "4096 stream-K")
    _check_sampled(c.A, c.B, D0, 4000, 31, "4096 plain")

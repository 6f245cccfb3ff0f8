"""GPU parity of the grouped (expert FC1) kernel against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl
from gpu_util import assert_bits_equal, assert_within_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


def run_grouped(A, Bs, offsets, sentinel=float("nan")):
    from blackwell_tensor_core_gb300 import ops
    dev = torch.device("cuda")
    Ad = A.to(dev)
    Bd = [b.to(dev) for b in Bs]
    off = torch.from_numpy(np.asarray(offsets, dtype=np.int32)).to(dev)
    N = Bs[0].shape[1]
    D = torch.full((A.shape[0], N), sentinel, dtype=A.dtype, device=dev)
    ops.grouped_gemm(Ad, Bd, off, out=D)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    return D.cpu(), st, word


def test_grouped_integer_exact_with_empty_and_ragged_groups():
    counts = [300, 0, 256, 1, 0, 511, 37]
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6000)
    K, N = 200, 600
    A = wl.randint_matrix(int(off[-1]), K, -2, 2, g)
    Bs = [wl.randint_matrix(K, N, -2, 2, g) for _ in counts]
    D, st, word = run_grouped(A, Bs, off)
    assert st == 0, hex(word)
    Dref, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off)
    assert_bits_equal(D, oracle.round_to(Dref, "bf16"), "grouped exact")


def test_grouped_random_within_bound_single_group_and_fp16():
    g = wl.generator(6001)
    for dtype in ("bf16", "fp16"):
        A = wl.normal_matrix(700, 264, 1.0, g, dtype)
        Bs = [wl.normal_matrix(264, 520, 0.5, g, dtype)]
        off = np.array([0, 700], np.int32)
        D, st, word = run_grouped(A, Bs, off)
        assert st == 0, hex(word)
        Dref, S = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off, dtype)
        assert_within_bound(D, Dref, S, "grouped G=1 " + dtype)


def test_grouped_more_than_64_groups():
    rng = np.random.default_rng(6002)
    counts = list(rng.integers(0, 40, 70))
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6003)
    K, N = 64, 256
    A = wl.randint_matrix(int(off[-1]), K, -2, 2, g)
    Bs = [wl.randint_matrix(K, N, -2, 2, g) for _ in counts]
    D, st, word = run_grouped(A, Bs, off)
    assert st == 0, hex(word)
    Dref, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off)
    assert_bits_equal(D, oracle.round_to(Dref, "bf16"), "grouped G=70")


def test_grouped_bad_offsets_are_reported_and_stay_in_bounds():
    g = wl.generator(6004)
    A = wl.normal_matrix(300, 64, 1.0, g)
    Bs = [wl.normal_matrix(64, 256, 1.0, g) for _ in range(3)]
    off = np.array([0, 200, 100, 300], np.int32)  # decreasing: breaks the contract
    D, st, word = run_grouped(A, Bs, off, sentinel=3.0)
    assert st == 1 and (word >> 56) == 2
    # clamped schedule: group 1 is empty, groups 0 and 2 still computed
    Dref0, S0 = oracle.gemm(wl.bits(A[:200]), wl.bits(Bs[0]))
    assert_within_bound(D[:200], Dref0, S0, "group 0")


def _check_grouped_sampled(c, D, seed):
    rng = np.random.default_rng(seed)
    Abits = wl.bits(c.A)
    for gi in range(c.G):
        r0, r1 = int(c.offsets[gi]), int(c.offsets[gi + 1])
        if r1 == r0:
            continue
        seams = [r0, r1 - 1, r0 + 255, r0 + 256, r0 + 511, r0 + 512]
        rows = np.concatenate([[min(r, r1 - 1) for r in seams], rng.integers(r0, r1, 58)])
        cols = np.concatenate([[0, c.N - 1, 255, 256, c.N // 2, 127], rng.integers(0, c.N, 58)])
        Dref, S = oracle.gemm_elements(Abits, wl.bits(c.Bs[gi]), rows, cols, c.in_dtype)
        assert_within_bound(D[rows, cols], Dref, S, "%s expert %d" % (c.name, gi))


def test_grouped_fc1_method_workload_sampled():
    c = wl.grouped_case()
    D, st, word = run_grouped(c.A, c.Bs, c.offsets)
    assert st == 0, hex(word)
    assert torch.isfinite(D.float()).all()
    _check_grouped_sampled(c, D, 13)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_grouped_fc2_method_workload_sampled(dtype):
    """Expert FC2 (down projection, K = 2048, N = 4096) over the FC1 case's
    token buckets, with the same grouped kernel."""
    c = wl.grouped_fc2_case(dtype=dtype)
    assert np.array_equal(c.offsets, wl.grouped_case().offsets)
    D, st, word = run_grouped(c.A, c.Bs, c.offsets)
    assert st == 0, hex(word)
    assert D.dtype == c.A.dtype and torch.isfinite(D.float()).all()
    _check_grouped_sampled(c, D, 14)


def test_grouped_fc1_fp16_sampled():
    c = wl.grouped_case(dtype="fp16")
    D, st, word = run_grouped(c.A, c.Bs, c.offsets)
    assert st == 0, hex(word)
    assert torch.isfinite(D.float()).all()
    _check_grouped_sampled(c, D, 15)


@pytest.mark.parametrize("counts", [[300, 0, 256, 1, 0, 511, 37], [16, 128, 129, 384, 100, 5]])
def test_grouped_swapped_group_ends_exact(counts, monkeypatch):
    """Group ends of at most 128 rows are computed with swapped operands
    (rows on the MMA's N); the result must be exact on integer inputs, the
    same as with swapping switched off, and rows outside every tile untouched."""
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6100 + len(counts))
    K, N = 192, 520
    A = wl.randint_matrix(int(off[-1]), K, -2, 2, g)
    Bs = [wl.randint_matrix(K, N, -2, 2, g) for _ in counts]
    Dref, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off)
    want = oracle.round_to(Dref, "bf16")
    monkeypatch.setenv("BWG_GROUPED_SWAP", "1")
    monkeypatch.setenv("BWG_GROUPED_1C", "1")  # swapped ends belong to the one-consumer kernel
    D, st, word = run_grouped(A, Bs, off)
    assert st == 0, hex(word)
    assert_bits_equal(D, want, "swapped ends")
    monkeypatch.delenv("BWG_GROUPED_SWAP")
    D2, st, word = run_grouped(A, Bs, off)
    assert st == 0, hex(word)
    assert_bits_equal(D2, want, "padded ends")


@pytest.mark.parametrize("one_consumer,sched", [("0", "clc"), ("0", "static"), ("1", "static")])
def test_grouped_both_kernels_exact(one_consumer, sched, monkeypatch):
    """Groups ending 1..511 rows into a 512-row unit (second consumer skipped
    at 256 rows or fewer), with dynamic and static scheduling, and the
    256-row kernel: all exact."""
    monkeypatch.setenv("BWG_GROUPED_1C", one_consumer)
    monkeypatch.setenv("BWG_SCHED", sched)
    counts = [1, 255, 256, 257, 511, 512, 513, 0, 700, 1030]
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6300)
    K, N = 128, 520
    A = wl.randint_matrix(int(off[-1]), K, -2, 2, g)
    Bs = [wl.randint_matrix(K, N, -2, 2, g) for _ in counts]
    Dref, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off)
    D, st, word = run_grouped(A, Bs, off)
    assert st == 0, hex(word)
    assert_bits_equal(D, oracle.round_to(Dref, "bf16"), "grouped consumers=%s" % one_consumer)


@pytest.mark.parametrize("swiglu", [False, True])
def test_grouped_dynamic_schedule(swiglu, monkeypatch):
    """Cluster-launch-control scheduling of the two-consumer grouped kernel:
    115 units (more than the pairs that fit at once), ragged and empty
    groups; exact without SwiGLU, within the SwiGLU bound with it."""
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_SCHED", "clc")
    counts = [1, 255, 256, 257, 511, 512, 513, 0, 700, 1030, 3000, 2048]
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6500)
    K, N = 64, 1040
    A = wl.randint_matrix(int(off[-1]), K, -2, 2, g)
    Bs = [wl.randint_matrix(K, N, -2, 2, g) for _ in counts]
    dev = torch.device("cuda")
    offd = torch.from_numpy(off).to(dev)
    out = torch.full((A.shape[0], N // 2 if swiglu else N), float("nan"), dtype=A.dtype, device=dev)
    ops.grouped_gemm(A.to(dev), [b.to(dev) for b in Bs], offd, out=out, swiglu=swiglu)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    if swiglu:
        Href, W = oracle.grouped_swiglu(wl.bits(A), [wl.bits(b) for b in Bs], off)
        bad = oracle.bound_violations(out.cpu().double().numpy(), Href, W)
        assert not bad.any(), "%d outside the SwiGLU bound" % bad.sum()
    else:
        Dref, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off)
        assert_bits_equal(out.cpu(), oracle.round_to(Dref, "bf16"), "grouped dynamic")


SHORT_END_COUNTS = [31, 512 + 32, 33, 63, 64, 65, 0, 100, 127, 128, 129, 1024 + 1, 512 + 64, 7]


@pytest.mark.parametrize("sched,swiglu", [("clc", False), ("static", False), ("clc", True)])
def test_grouped_short_group_ends(sched, swiglu, monkeypatch):
    """Two-consumer kernel, group ends of 1..129 rows (31, 32, 33, 63, 64,
    65, 100, 127, 128, 129 and 1 past a multiple of 512), an empty group, and
    a last group of 7 rows whose 128-row A boxes reach past the end of A:
    exact on integer inputs, within the SwiGLU bound with the fused epilogue."""
    from blackwell_tensor_core_gb300 import ops
    monkeypatch.setenv("BWG_SCHED", sched)
    counts = SHORT_END_COUNTS
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6700)
    K, N = 192, 528
    A = wl.randint_matrix(int(off[-1]), K, -2, 2, g)
    Bs = [wl.randint_matrix(K, N, -2, 2, g) for _ in counts]
    dev = torch.device("cuda")
    offd = torch.from_numpy(off).to(dev)
    out = torch.full((A.shape[0], N // 2 if swiglu else N), float("nan"), dtype=A.dtype, device=dev)
    ops.grouped_gemm(A.to(dev), [b.to(dev) for b in Bs], offd, out=out, swiglu=swiglu)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    if swiglu:
        Href, W = oracle.grouped_swiglu(wl.bits(A), [wl.bits(b) for b in Bs], off)
        bad = oracle.bound_violations(out.cpu().double().numpy(), Href, W)
        assert not bad.any(), "%d outside the SwiGLU bound" % bad.sum()
    else:
        Dref, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off)
        assert_bits_equal(out.cpu(), oracle.round_to(Dref, "bf16"), "short group ends %s" % sched)

"""GPU parity of the grouped FC1 kernel with the fused SwiGLU epilogue
(H = silu(gate) * up, B_g = [gate | up]) against the CPU oracle.

Tolerance (derived in the oracle's docstring from the GEMM bound):
    |H - H_ref| <= 2^-7 |H_ref| + 1e-3 W,
    W = 1.1 |up| S_gate + |silu(gate)| S_up + 1.1e-3 S_gate S_up."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


def run_swiglu(A, Bs, offsets, sentinel=float("nan")):
    from blackwell_tensor_core_gb300 import ops
    dev = torch.device("cuda")
    Ad = A.to(dev)
    Bd = [b.to(dev) for b in Bs]
    off = torch.from_numpy(np.asarray(offsets, dtype=np.int32)).to(dev)
    N = Bs[0].shape[1]
    H = torch.full((A.shape[0], N // 2), sentinel, dtype=A.dtype, device=dev)
    ops.grouped_gemm(Ad, Bd, off, out=H, swiglu=True)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    return H.cpu(), st, word


def assert_swiglu_bound(H, Href, W, what):
    Hv = H.double().numpy() if isinstance(H, torch.Tensor) else np.asarray(H, np.float64)
    bad = oracle.bound_violations(Hv, Href, W)
    if bad.any():
        idx = [tuple(i) for i in np.argwhere(bad)[:5]]
        raise AssertionError("%s: %d of %d outside the bound; first %s" % (
            what, int(bad.sum()), bad.size,
            ", ".join("%s got %r want %r W %r" % (i, Hv[i], Href[i], W[i]) for i in idx)))


@pytest.mark.parametrize("one_consumer", ["0", "1"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_swiglu_ragged_groups_within_bound(one_consumer, dtype, monkeypatch):
    """Empty, 1-row, 255..513-row and multi-tile groups; N/2 = 200 output
    columns (a ragged column tile); K = 200 (a ragged k-block)."""
    monkeypatch.setenv("BWG_GROUPED_1C", one_consumer)
    counts = [300, 0, 256, 1, 0, 511, 37, 513, 1030]
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6400)
    K, N = 200, 400
    A = wl.normal_matrix(int(off[-1]), K, 1.0, g, dtype)
    Bs = [wl.normal_matrix(K, N, 0.15, g, dtype) for _ in counts]
    H, st, word = run_swiglu(A, Bs, off)
    assert st == 0, hex(word)
    Href, W = oracle.grouped_swiglu(wl.bits(A), [wl.bits(b) for b in Bs], off, dtype)
    assert_swiglu_bound(H, Href, W, "swiglu %s consumers=%s" % (dtype, one_consumer))


@pytest.mark.parametrize("row_tiles", [11, 12])
@pytest.mark.parametrize("no_split", ["0", "1"])
def test_swiglu_last_wave_cuts(row_tiles, no_split, monkeypatch):
    """8 column tiles (N/2 = 1024) x 11 or 12 row units of 512: on 76 CTA
    pairs the last wave is cut into quarters (88 units) or halves (96), or
    not at all with BWG_NO_TAIL_SPLIT=1; every cut must give the same H."""
    monkeypatch.setenv("BWG_NO_TAIL_SPLIT", no_split)
    counts = [1536, 1124, 2041, 300] if row_tiles == 11 else [1536, 1124, 2041, 812]
    assert sum((c + 511) // 512 for c in counts) == row_tiles
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6410 + row_tiles)
    K, N = 64, 2048
    A = wl.normal_matrix(int(off[-1]), K, 1.0, g)
    Bs = [wl.normal_matrix(K, N, 0.25, g) for _ in counts]
    H, st, word = run_swiglu(A, Bs, off)
    assert st == 0, hex(word)
    Href, W = oracle.grouped_swiglu(wl.bits(A), [wl.bits(b) for b in Bs], off)
    assert_swiglu_bound(H, Href, W, "swiglu cut, %d row units, no_split=%s" % (row_tiles, no_split))


def test_swiglu_integer_inputs_and_large_gates():
    """Integer inputs make gate and up exact in FP32, so the only error left
    is the activation and one rounding: within 2^-7 |H_ref| alone (W is
    large here, so check the relative part by itself)."""
    counts = [130, 600, 5]
    off = wl.offsets_from_counts(counts)
    g = wl.generator(6420)
    K, N = 128, 256
    A = wl.randint_matrix(int(off[-1]), K, -2, 2, g)
    Bs = [wl.randint_matrix(K, N, -2, 2, g) for _ in counts]
    H, st, word = run_swiglu(A, Bs, off)
    assert st == 0, hex(word)
    Href, _ = oracle.grouped_swiglu(wl.bits(A), [wl.bits(b) for b in Bs], off)
    Hv = H.double().numpy()
    tiny = np.abs(Href) < 1e-30  # far-negative gates: both sides are (signed) zero or tiny
    err = np.abs(Hv - Href)
    assert (err[~tiny] <= 2.0 ** -8 * np.abs(Href[~tiny])).all()
    assert (np.abs(Hv[tiny]) < 1e-30).all()


def test_swiglu_fc1_method_workload_sampled():
    """The grouped FC1 workload (32 experts, 32768 rows, K = 4096, B_g =
    [gate | up] with 2048 columns each): H sampled at every expert's first,
    last and 256/512-row seam rows and at column-tile seams."""
    c = wl.grouped_case()
    H, st, word = run_swiglu(c.A, c.Bs, c.offsets)
    assert st == 0, hex(word)
    assert torch.isfinite(H.float()).all()
    I_out = c.N // 2
    rng = np.random.default_rng(17)
    Abits = wl.bits(c.A)
    for gi in range(c.G):
        r0, r1 = int(c.offsets[gi]), int(c.offsets[gi + 1])
        if r1 == r0:
            continue
        seams = [r0, r1 - 1, r0 + 255, r0 + 256, r0 + 511, r0 + 512]
        rows = np.concatenate([[min(r, r1 - 1) for r in seams], rng.integers(r0, r1, 34)])
        cols = np.concatenate([[0, 63, 64, 127, 128, I_out - 1], rng.integers(0, I_out, 34)])
        Href, W = oracle.swiglu_elements(Abits, wl.bits(c.Bs[gi]), rows, cols)
        assert_swiglu_bound(H[rows, cols], Href, W, "expert %d" % gi)


def test_swiglu_zero_k_and_argument_errors():
    from blackwell_tensor_core_gb300 import ops
    dev = torch.device("cuda")
    off = torch.tensor([0, 40, 100], dtype=torch.int32, device=dev)
    A = torch.empty((100, 0), dtype=torch.bfloat16, device=dev)
    Bs = [torch.empty((0, 64), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    H = torch.full((100, 32), 7.0, dtype=torch.bfloat16, device=dev)
    ops.grouped_gemm(A, Bs, off, out=H, swiglu=True)
    torch.cuda.synchronize()
    assert (H == 0).all()
    # N = 24: the up block would start at column 12, not on a 16-byte boundary
    A = torch.zeros((100, 64), dtype=torch.bfloat16, device=dev)
    Bs = [torch.zeros((64, 24), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    H = torch.zeros((100, 12), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ops.BwgError) as e:
        ops.grouped_gemm(A, Bs, off, out=H, swiglu=True)
    assert e.value.status == 2

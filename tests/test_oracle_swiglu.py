"""Pins for the oracle's SwiGLU (H = silu(gate) * up on a [gate | up] GEMM).

Each test checks it against something other than itself: closed forms of the
logistic function, a library routine (scipy's expit), an exact integer GEMM
feeding known activations, and the grouped and single-element forms against
the whole-matrix form.  A swapped gate/up, a dropped factor, a wrong sign in
the exponent or a wrong column offset each fail at least one of them."""
import math

import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl


def _pairs(gate, up):
    gate = np.atleast_2d(np.asarray(gate, dtype=np.float64))
    up = np.atleast_2d(np.asarray(up, dtype=np.float64))
    return np.concatenate([gate, up], axis=1)


def test_closed_forms_of_silu():
    # silu(0) = 0; sigmoid(ln 3) = 3/4; silu(x) = x once e^-x is below half an
    # ulp of 1; silu(-x) = -x e^-x / (1 + e^-x)
    x = np.array([0.0, math.log(3.0), 40.0, -40.0, 1.0])
    H = oracle.swiglu(_pairs(x, np.ones_like(x)))[0]
    assert H[0] == 0.0
    assert H[1] == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    assert H[2] == 40.0
    assert H[3] == pytest.approx(-40.0 * math.exp(-40.0) / (1.0 + math.exp(-40.0)), rel=1e-14)
    assert H[4] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


def test_silu_odd_part_is_identity():
    # silu(x) - silu(-x) = x (sigma(x) + sigma(-x)) = x, for every x
    x = np.linspace(-30.0, 30.0, 601)
    Hp = oracle.swiglu(_pairs(x, np.ones_like(x)))[0]
    Hm = oracle.swiglu(_pairs(-x, np.ones_like(x)))[0]
    assert np.allclose(Hp - Hm, x, rtol=1e-13, atol=1e-13)


def test_silu_matches_scipy_expit():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    x = rng.normal(0.0, 8.0, 4000)
    u = rng.normal(0.0, 2.0, 4000)
    H = oracle.swiglu(_pairs(x, u))[0]
    assert np.allclose(H, x * special.expit(x) * u, rtol=1e-13, atol=0.0)


def test_far_negative_gate_gives_signed_zero_not_nan():
    x = np.array([-800.0, -1e6])
    H = oracle.swiglu(_pairs(x, np.array([2.0, -3.0])))[0]
    assert not np.isnan(H).any() and np.all(H == 0.0)


def test_gate_is_the_first_column_block():
    """Integer GEMM whose up block is identically 1 and whose gate block is
    known: H must be silu(gate), not gate * silu(1) or silu(1)."""
    g = wl.generator(31)
    M, K, I = 9, 6, 5
    A = wl.randint_matrix(M, K, -2, 2, g)
    A[:, 0] = 1  # column 0 of A is all ones
    Bg = wl.randint_matrix(K, I, -2, 2, g)
    Bu = torch.zeros((K, I), dtype=torch.bfloat16)
    Bu[0, :] = 1  # up = A[:, 0] = 1
    B = torch.cat([Bg, Bu], dim=1)
    D, S = oracle.gemm(wl.bits(A), wl.bits(B))
    H = oracle.swiglu(D)
    gate = A.to(torch.int64).numpy() @ Bg.to(torch.int64).numpy()
    assert np.allclose(H, gate / (1.0 + np.exp(-gate.astype(np.float64))), rtol=1e-15, atol=0.0)


def test_large_gate_passes_up_through_times_gate():
    """Gate >= 40 makes silu exact (= gate) in double: H = gate * up exactly."""
    M, K, I = 4, 3, 3
    A = torch.tensor([[20, 1, -2], [20, 2, 1], [21, -1, 0], [22, 0, 2]], dtype=torch.bfloat16)
    Bg = torch.tensor([[2, 2, 3], [0, 1, 0], [0, 0, 1]], dtype=torch.bfloat16)
    Bu = torch.tensor([[0, 1, 0], [1, 0, -1], [2, 1, 1]], dtype=torch.bfloat16)
    D, _ = oracle.gemm(wl.bits(A), wl.bits(torch.cat([Bg, Bu], dim=1)))
    a = A.to(torch.int64).numpy()
    gate = a @ Bg.to(torch.int64).numpy()
    up = a @ Bu.to(torch.int64).numpy()
    assert gate.min() >= 40
    assert np.array_equal(oracle.swiglu(D), (gate * up).astype(np.float64))
    assert M == 4 and K == 3 and I == 3


def test_grouped_and_elements_agree_with_whole_matrix_form():
    counts = [7, 0, 12, 1, 5]
    off = wl.offsets_from_counts(counts)
    g = wl.generator(32)
    K, I = 40, 24
    A = wl.normal_matrix(int(off[-1]), K, 1.0, g)
    Bs = [wl.normal_matrix(K, 2 * I, 0.3, g) for _ in counts]
    H, W = oracle.grouped_swiglu(wl.bits(A), [wl.bits(b) for b in Bs], off)
    assert H.shape == (int(off[-1]), I) and W.shape == H.shape
    for e in range(len(counts)):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        D, S = oracle.gemm(wl.bits(A[r0:r1]), wl.bits(Bs[e]))
        assert np.array_equal(H[r0:r1], oracle.swiglu(D))
        rows = np.arange(r0, r1)
        cols = np.arange(r1 - r0) % I
        He, We = oracle.swiglu_elements(wl.bits(A), wl.bits(Bs[e]), rows, cols)
        assert np.array_equal(He, H[rows, cols])
        assert np.array_equal(We, W[rows, cols])


def test_silu_slope_bound_used_by_the_tolerance():
    """The tolerance carries a gate error through silu with |silu'| < 1.1:
    check the slope of the oracle's silu on a fine grid."""
    x = np.linspace(-60.0, 60.0, 240001)
    s = oracle.swiglu(_pairs(x, np.ones_like(x)))[0]
    slope = np.diff(s) / np.diff(x)
    assert np.abs(slope).max() < 1.1
    assert np.abs(slope).max() > 1.09  # the maximum, near x = 2.4, is about 1.0998


def test_bound_weight_catches_planted_errors():
    """Rounding H to BF16 stays inside the bound; an error just past the
    bound is caught."""
    g = wl.generator(33)
    A = wl.randint_matrix(16, 8, -2, 2, g)
    B = wl.randint_matrix(8, 32, -2, 2, g)
    D, S = oracle.gemm(wl.bits(A), wl.bits(B))
    H, silu = oracle.swiglu(D, with_silu=True)
    W = oracle.swiglu_weight(D, S, silu)
    Hr = torch.from_numpy(H).to(torch.bfloat16).double().numpy()
    assert not oracle.bound_violations(Hr, H, W).any()
    bad = H + np.sign(H) * (2.0 ** -6 * np.abs(H) + 1e-3 * W + 1e-6)
    big = np.abs(H) > 1.0
    assert oracle.bound_violations(bad, H, W)[big].all()

"""Pins for the CPU oracle: each test checks it against something other than
itself (library conversions, exact integer matmul, closed forms, exact rational
brute force, structured matrices), chosen so a dropped term, a wrong sign or
index, or a transposed operand fails at least one of them."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl


def _bf16(x):
    return wl.bits(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def _fp16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


# --- format decoding -------------------------------------------------------

def test_decode_bf16_all_patterns_match_torch():
    pats = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode(pats, "bf16")
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_fp16_all_patterns_match_numpy():
    pats = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode(pats, "fp16")
    ref = pats.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_known_values():
    assert oracle.decode(np.array([0x3F80, 0xC000, 0x0000, 0x8000], np.uint16), "bf16").tolist() == [1.0, -2.0, 0.0, -0.0]
    assert oracle.decode(np.array([0x3C00, 0x7BFF, 0x0001, 0x0400], np.uint16), "fp16").tolist() == [
        1.0, 65504.0, 2.0 ** -24, 2.0 ** -14]


# --- output rounding --------------------------------------------------------

def test_round_bf16_matches_torch_on_binary32_values():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(1000.0),
        np.float32(1.0) + np.arange(-300, 300, dtype=np.float32) * np.float32(2.0 ** -9),  # ties
        np.array([0.0, -0.0, 3.0e38, -3.0e38, 1e-40, 255.0, 257.0, 259.0, 2047.0, 2049.0], np.float32),
    ])
    ours = oracle.round_to(x.astype(np.float64), "bf16")
    ref = wl.bits(torch.from_numpy(x).to(torch.bfloat16))
    assert np.array_equal(ours, ref)


def test_round_fp16_matches_numpy():
    rng = np.random.default_rng(8)
    x = np.concatenate([
        rng.standard_normal(20000) * 300.0,
        rng.standard_normal(2000) * 1e-5,  # subnormals
        1.0 + np.arange(-300, 300) * 2.0 ** -11,  # ties at 1.0
        np.array([65504.0, 65519.0, 65520.0, 70000.0, -65520.0, 2.0 ** -25, 3 * 2.0 ** -26, 0.0, -0.0]),
    ])
    ours = oracle.round_to(x, "fp16")
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# --- structured products ----------------------------------------------------

def test_identity_left_and_right():
    g = wl.generator(11)
    B = wl.normal_matrix(48, 37, 1.0, g)
    I48 = torch.eye(48).to(torch.bfloat16)
    D, S = oracle.gemm(wl.bits(I48), wl.bits(B))
    assert np.array_equal(D, B.double().numpy())
    assert np.array_equal(S, B.double().abs().numpy())
    A = wl.normal_matrix(29, 48, 1.0, g)
    D, _ = oracle.gemm(wl.bits(A), wl.bits(I48))
    assert np.array_equal(D, A.double().numpy())


def test_permutation_rows_and_columns():
    rng = np.random.default_rng(3)
    g = wl.generator(12)
    B = wl.normal_matrix(40, 23, 1.0, g)
    p = rng.permutation(40)
    P = np.zeros((40, 40), np.float32)
    P[np.arange(40), p] = 1.0  # (P B)[i] = B[p[i]]
    D, _ = oracle.gemm(_bf16(P), wl.bits(B))
    assert np.array_equal(D, B.double().numpy()[p])
    A = wl.normal_matrix(17, 40, 1.0, g)
    q = rng.permutation(40)
    Q = np.zeros((40, 40), np.float32)
    Q[q, np.arange(40)] = 1.0  # (A Q)[:, j] = A[:, q[j]]
    D, _ = oracle.gemm(wl.bits(A), _bf16(Q))
    assert np.array_equal(D, A.double().numpy()[:, q])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_small_integers_exact_against_integer_matmul(dtype):
    g = wl.generator(13)
    A = wl.randint_matrix(37, 71, -2, 2, g, dtype)
    B = wl.randint_matrix(71, 53, -2, 2, g, dtype)
    D, S = oracle.gemm(wl.bits(A), wl.bits(B), dtype)
    Ai = A.to(torch.int64).numpy()
    Bi = B.to(torch.int64).numpy()
    assert np.array_equal(D, (Ai @ Bi).astype(np.float64))
    assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


def test_strided_buffers_ignore_padding():
    g = wl.generator(14)
    A = wl.randint_matrix(19, 40, -2, 2, g)   # lda = 40, K = 33
    B = wl.randint_matrix(33, 64, -2, 2, g)   # ldb = 64, N = 27
    D, _ = oracle.gemm_strided(wl.bits(A), wl.bits(B), 19, 27, 33)
    ref = A[:, :33].to(torch.int64).numpy() @ B[:, :27].to(torch.int64).numpy()
    assert np.array_equal(D, ref.astype(np.float64))


def test_all_ones_gives_K():
    for K in (1, 7, 64, 300):
        A = torch.ones(5, K).to(torch.bfloat16)
        B = torch.ones(K, 9).to(torch.bfloat16)
        D, S = oracle.gemm(wl.bits(A), wl.bits(B))
        assert np.all(D == K) and np.all(S == K)


def test_rank_one_closed_form_with_signs():
    rng = np.random.default_rng(4)
    choices = np.array([1.0, -1.0, 2.0, -2.0, 0.5, -0.5, 4.0, -0.25])
    u, x = rng.choice(choices, 13), rng.choice(choices, 31)
    y, v = rng.choice(choices, 31), rng.choice(choices, 11)
    A = np.outer(u, x)
    B = np.outer(y, v)
    D, S = oracle.gemm(_bf16(A), _bf16(B))
    assert np.array_equal(D, np.outer(u, v) * float(np.dot(x, y)))
    assert np.array_equal(S, np.outer(np.abs(u), np.abs(v)) * float(np.dot(np.abs(x), np.abs(y))))


def test_brute_force_tiny_shapes_exact_rationals():
    rng = np.random.default_rng(5)
    for M in range(1, 5):
        for N in range(1, 5):
            for K in range(1, 5):
                A = _bf16(rng.standard_normal((M, K)))
                B = _bf16(rng.standard_normal((K, N)))
                av = torch.from_numpy(A.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
                bv = torch.from_numpy(B.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
                D, S = oracle.gemm(A, B)
                for i in range(M):
                    for j in range(N):
                        terms = [Fraction(float(av[i, k])) * Fraction(float(bv[k, j])) for k in range(K)]
                        exact = sum(terms, Fraction(0))
                        sabs = sum((abs(t) for t in terms), Fraction(0))
                        # K <= 4 products of 8-bit significands: the double sum is exact
                        assert Fraction(D[i, j]) == exact
                        assert Fraction(S[i, j]) == sabs


def test_elements_against_numpy_float64():
    g = wl.generator(15)
    A = wl.normal_matrix(33, 90, 1.0, g)
    B = wl.normal_matrix(90, 45, 1.0, g)
    ref = A.double().numpy() @ B.double().numpy()
    rng = np.random.default_rng(6)
    I = rng.integers(0, 33, 500)
    J = rng.integers(0, 45, 500)
    D, S = oracle.gemm_elements(wl.bits(A), wl.bits(B), I, J)
    assert np.allclose(D, ref[I, J], rtol=1e-13, atol=1e-13)
    assert np.all(S >= np.abs(D))
    Dr, _ = oracle.gemm(wl.bits(A), wl.bits(B))
    assert np.allclose(Dr, ref, rtol=1e-13, atol=1e-13)


def test_sign_flip_and_absolute_sum():
    g = wl.generator(16)
    A = wl.normal_matrix(21, 34, 1.0, g)
    B = wl.normal_matrix(34, 18, 1.0, g)
    D, S = oracle.gemm(wl.bits(A), wl.bits(B))
    Dn, Sn = oracle.gemm(wl.bits(-A), wl.bits(B))
    Da, _ = oracle.gemm(wl.bits(A.abs()), wl.bits(B.abs()))
    assert np.array_equal(Dn, -D)
    assert np.array_equal(Sn, S)
    assert np.array_equal(Da, S)


def test_grouped_scaled_identity_weights_and_empty_groups():
    counts = [3, 0, 5, 1, 0, 4]
    off = wl.offsets_from_counts(counts)
    G, K = len(counts), 24
    g = wl.generator(17)
    A = wl.normal_matrix(int(off[-1]), K, 1.0, g)
    Bs = [(torch.eye(K) * (e + 1)).to(torch.bfloat16) for e in range(G)]
    D, S = oracle.grouped_gemm(wl.bits(A), [wl.bits(b) for b in Bs], off)
    a = A.double().numpy()
    for e in range(G):
        r0, r1 = off[e], off[e + 1]
        assert np.array_equal(D[r0:r1], a[r0:r1] * (e + 1))
        assert np.array_equal(S[r0:r1], np.abs(a[r0:r1]) * (e + 1))


def test_grouped_single_group_equals_dense():
    g = wl.generator(18)
    A = wl.randint_matrix(50, 30, -2, 2, g)
    B = wl.randint_matrix(30, 20, -2, 2, g)
    D, _ = oracle.grouped_gemm(wl.bits(A), [wl.bits(B)], np.array([0, 50], np.int32))
    ref = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy()
    assert np.array_equal(D, ref.astype(np.float64))


def test_bound_catches_planted_errors():
    Dref = np.array([100.0, -100.0, 0.0, 1.0])
    S = np.array([200.0, 200.0, 10.0, 1.0])
    ok = Dref.copy()
    assert not oracle.bound_violations(ok, Dref, S).any()
    bad = Dref + np.array([0.0, 0.0, 0.0, 0.5])
    assert oracle.bound_violations(bad, Dref, S).tolist() == [False, False, False, True]
    # 2^-7 * 100 + 1e-3 * 200 = 0.98125: just inside and just outside
    assert not oracle.bound_violations(np.array([100.98]), np.array([100.0]), np.array([200.0])).any()
    assert oracle.bound_violations(np.array([100.99]), np.array([100.0]), np.array([200.0])).all()
    assert oracle.bound_violations(np.array([np.nan]), np.array([0.0]), np.array([1.0])).all()


def test_workload_generators_are_seeded_and_shaped():
    c1, c1b = wl.tile_case(), wl.tile_case()
    assert torch.equal(c1.A, c1b.A) and torch.equal(c1.B, c1b.B)
    assert c1.A.shape == (256, 512) and c1.B.shape == (512, 256)
    assert set(torch.unique(c1.A.float()).tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    counts = wl.expert_counts(4096, 8, 32, wl.generator(1005))
    assert counts.sum() == 32768 and len(counts) == 32
    # FC2 runs over the FC1 case's token buckets
    fc1 = wl.grouped_case(experts=4, N=16, K=16)
    fc2 = wl.grouped_fc2_case(experts=4, N=16, K=16)
    assert np.array_equal(fc1.offsets, fc2.offsets) and fc2.A.shape == (fc1.total, 16)
    assert wl.square_case(n=64, dtype="fp16").A.dtype == torch.float16

"""CPU oracle for D = A x B with BF16/FP16 inputs (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
in ``blackwell_tensor_core_gb300`` and never imports it; the two meet only in
the seeded input generators, which hold none of the method's arithmetic.

The arithmetic lives in ``gemm_oracle.c`` (plain C, FP64): a triple loop
written from the per-element definition on the page "B200 的 2CTA 怎样调优",
section 七 (acc = sum_k A[i,k]*B[k,j], then convert).  This module only builds
that file with gcc, loads it with ctypes and marshals numpy arrays.

Acceptance (the method's stated bound, one element at a time):
    |D - D_ref| <= 2^-7 * |D_ref| + 1e-3 * S,   S = sum_k |A[i,k]*B[k,j]|
and bit-exact agreement where inputs are integer-valued and every partial sum
is exactly representable in binary32.

SwiGLU (``swiglu``, ``grouped_swiglu``, ``swiglu_elements``): H = silu(gate) *
up on the FP64 GEMM of a [gate | up] weight, computed in ``oracle_swiglu``.
Its acceptance bound is the GEMM's carried through the activation:
    |H - H_ref| <= 2^-7 |H_ref| + 1e-3 * W,
    W = 1.1 |up| S_gate + |silu(gate)| S_up + 1.1e-3 S_gate S_up,
because an accumulator error e_g <= 1e-3 S_gate moves silu(gate) by at most
1.1 e_g (|silu'| < 1.1 everywhere), an error e_u <= 1e-3 S_up moves the
product by |silu(gate)| e_u, the cross term is their product, and the final
rounding to BF16/FP16 with the activation's own evaluation error stays inside
2^-7 |H_ref|.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

IN_BF16 = 0
IN_FP16 = 1
_DTYPES = {"bf16": IN_BF16, "fp16": IN_FP16}


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into liboracle.so with gcc (OpenMP, no fast-math)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            lib.oracle_gemm_rows.argtypes = [u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                             ctypes.c_int, dp, dp]
            lib.oracle_gemm_rows.restype = None
            lib.oracle_gemm_elements.argtypes = [u16p, u16p, ctypes.c_int, ctypes.c_int, ctypes.c_long,
                                                 ctypes.c_long, lp, lp, ctypes.c_long, dp, dp]
            lib.oracle_gemm_elements.restype = None
            lib.oracle_grouped_gemm.argtypes = [u16p, ctypes.POINTER(u16p), ctypes.POINTER(ctypes.c_int),
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                dp, dp]
            lib.oracle_grouped_gemm.restype = None
            lib.oracle_swiglu.argtypes = [dp, ctypes.c_long, ctypes.c_int, dp, dp]
            lib.oracle_swiglu.restype = None
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_fp16_to_double.restype = ctypes.c_double
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_round_fp16.argtypes = [ctypes.c_double]
            lib.oracle_round_fp16.restype = ctypes.c_uint16
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def _u16(a: np.ndarray) -> np.ndarray:
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are 16-bit patterns (numpy uint16), got %s" % a.dtype)
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Run later calls on `n` OpenMP threads (timing aid; results do not change)."""
    _load().oracle_set_num_threads(int(n))


def decode(bits: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    """Exact value of each 16-bit pattern as float64 (one C call per element)."""
    lib = _load()
    f = lib.oracle_fp16_to_double if dtype == "fp16" else lib.oracle_bf16_to_double
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([f(int(x)) for x in flat], dtype=np.float64).reshape(np.shape(bits))


def round_to(values: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to bf16/fp16 bit patterns (nearest, ties to even)."""
    lib = _load()
    f = lib.oracle_round_fp16 if dtype == "fp16" else lib.oracle_round_bf16
    flat = np.asarray(values, dtype=np.float64).ravel()
    return np.array([f(float(x)) for x in flat], dtype=np.uint16).reshape(np.shape(values))


def gemm(A: np.ndarray, B: np.ndarray, dtype: str = "bf16", rows: tuple[int, int] | None = None):
    """D_ref and S for D = A x B.

    A: uint16 [M, >=K] row-major bit patterns (lda = A.shape[1] after slicing is
    not supported: pass the full buffer with ``K`` implied by B).  B: uint16
    [K, >=N].  Returns float64 arrays (D, S) of shape [rows, N].
    """
    A = np.ascontiguousarray(_u16(A))
    B = np.ascontiguousarray(_u16(B))
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: A is %s, B is %s" % (A.shape, B.shape))
    r0, r1 = rows if rows is not None else (0, M)
    D = np.empty((r1 - r0, N), dtype=np.float64)
    S = np.empty((r1 - r0, N), dtype=np.float64)
    _load().oracle_gemm_rows(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), _DTYPES[dtype],
                             M, N, K, K, N, r0, r1, _ptr(D, ctypes.c_double), _ptr(S, ctypes.c_double))
    return D, S


def gemm_strided(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, dtype: str = "bf16"):
    """Like gemm() but A is [M, lda] and B is [K, ldb] with padding columns ignored."""
    A = np.ascontiguousarray(_u16(A))
    B = np.ascontiguousarray(_u16(B))
    lda, ldb = A.shape[1], B.shape[1]
    if A.shape[0] < M or lda < K or B.shape[0] < K or ldb < N:
        raise ValueError("buffers smaller than the problem")
    D = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_rows(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), _DTYPES[dtype],
                             M, N, K, lda, ldb, 0, M, _ptr(D, ctypes.c_double), _ptr(S, ctypes.c_double))
    return D, S


def gemm_elements(A: np.ndarray, B: np.ndarray, I: np.ndarray, J: np.ndarray, dtype: str = "bf16"):
    """D_ref[I[t], J[t]] and S at a list of single outputs (one dot product each)."""
    A = np.ascontiguousarray(_u16(A))
    B = np.ascontiguousarray(_u16(B))
    K = A.shape[1]
    if B.shape[0] != K:
        raise ValueError("inner dimensions differ")
    I = np.ascontiguousarray(I, dtype=np.int64)
    J = np.ascontiguousarray(J, dtype=np.int64)
    if I.shape != J.shape:
        raise ValueError("index lists differ in length")
    D = np.empty(I.shape, dtype=np.float64)
    S = np.empty(I.shape, dtype=np.float64)
    _load().oracle_gemm_elements(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16), _DTYPES[dtype], K,
                                 A.shape[1], B.shape[1], _ptr(I, ctypes.c_long), _ptr(J, ctypes.c_long),
                                 I.size, _ptr(D, ctypes.c_double), _ptr(S, ctypes.c_double))
    return D, S


def grouped_gemm(A: np.ndarray, Bs: list, offsets: np.ndarray, dtype: str = "bf16"):
    """Grouped product: rows offsets[g]:offsets[g+1] of A times Bs[g]."""
    A = np.ascontiguousarray(_u16(A))
    G = len(Bs)
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    if offsets.shape != (G + 1,):
        raise ValueError("offsets needs G+1 entries")
    K = A.shape[1]
    N = Bs[0].shape[1] if G else 0
    Bs = [np.ascontiguousarray(_u16(b)) for b in Bs]
    for b in Bs:
        if b.shape != (K, N):
            raise ValueError("every weight matrix must be [K, N]")
    total = int(offsets[-1])
    D = np.zeros((total, N), dtype=np.float64)
    S = np.zeros((total, N), dtype=np.float64)
    arr = (ctypes.POINTER(ctypes.c_uint16) * max(G, 1))(*[_ptr(b, ctypes.c_uint16) for b in Bs])
    _load().oracle_grouped_gemm(_ptr(A, ctypes.c_uint16), arr, _ptr(offsets, ctypes.c_int), G, N, K,
                                _DTYPES[dtype], _ptr(D, ctypes.c_double), _ptr(S, ctypes.c_double))
    return D, S


def bound_violations(D: np.ndarray, D_ref: np.ndarray, S: np.ndarray,
                     rel: float = 2.0 ** -7, abs_frac: float = 1e-3) -> np.ndarray:
    """Boolean mask of elements outside |D - D_ref| <= rel*|D_ref| + abs_frac*S."""
    D = np.asarray(D, dtype=np.float64)
    err = np.abs(D - D_ref)
    lim = rel * np.abs(D_ref) + abs_frac * S
    return ~(err <= lim)  # NaN counts as a violation


def swiglu(D: np.ndarray, with_silu: bool = False):
    """H = silu(gate) * up for D = [gate | up] ([rows, 2I] float64) -> [rows, I].

    With ``with_silu`` also returns silu(gate) (for the error bound)."""
    D = np.ascontiguousarray(D, dtype=np.float64)
    rows, n2 = D.shape
    if n2 % 2:
        raise ValueError("D must have an even number of columns: [gate | up]")
    I = n2 // 2
    H = np.empty((rows, I), dtype=np.float64)
    silu = np.empty((rows, I), dtype=np.float64)
    _load().oracle_swiglu(_ptr(D, ctypes.c_double), rows, I, _ptr(H, ctypes.c_double),
                          _ptr(silu, ctypes.c_double))
    return (H, silu) if with_silu else H


def swiglu_weight(D: np.ndarray, S: np.ndarray, silu: np.ndarray) -> np.ndarray:
    """W of the SwiGLU bound (module docstring) from D = [gate | up], S and silu(gate)."""
    I = D.shape[1] // 2
    up, s_gate, s_up = D[:, I:], S[:, :I], S[:, I:]
    return 1.1 * np.abs(up) * s_gate + np.abs(silu) * s_up + 1.1e-3 * s_gate * s_up


def grouped_swiglu(A: np.ndarray, Bs: list, offsets: np.ndarray, dtype: str = "bf16"):
    """Grouped FC1 with SwiGLU: H [rows, N/2] and its bound weight W."""
    D, S = grouped_gemm(A, Bs, offsets, dtype)
    H, silu = swiglu(D, with_silu=True)
    return H, swiglu_weight(D, S, silu)


def swiglu_elements(A: np.ndarray, B: np.ndarray, I: np.ndarray, J: np.ndarray, dtype: str = "bf16"):
    """H[I[t], J[t]] and W for B = [gate | up] ([K, 2*width]), one pair of dot products each."""
    width = B.shape[1] // 2
    J = np.asarray(J, dtype=np.int64)
    I = np.asarray(I, dtype=np.int64)
    Dg, Sg = gemm_elements(A, B, I, J, dtype)
    Du, Su = gemm_elements(A, B, I, J + width, dtype)
    D = np.stack([Dg, Du], axis=1)
    S = np.stack([Sg, Su], axis=1)
    H, silu = swiglu(D, with_silu=True)
    return H[:, 0], swiglu_weight(D, S, silu)[:, 0]

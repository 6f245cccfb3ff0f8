"""Every output of the method's full-size workloads against the CPU oracle.

The dense products run through gemm_bf16 / gemm_fp16 exactly as the
benchmark calls them (dense row-major operands, lda = K, ldb = ldd = N,
default kernel choice); the expert products through grouped_gemm_bf16 /
grouped_gemm_swiglu_bf16 as the benchmark's variants call them.  The oracle
(plain FP64 triple loop, "B200 的 2CTA 怎样调优" section 七: acc = sum_k a*b,
then convert) runs in blocks of rows so that D_ref and S stay small, and every
element must satisfy the stated bound
    |D - D_ref| <= 2^-7 |D_ref| + 1e-3 sum_k |a_ik b_kj|
(for SwiGLU the same bound carried through the activation, see oracle.swiglu).
These take minutes of host time; the sampled tests elsewhere are the quick
checks of the same workloads."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl
from gpu_util import assert_within_bound, gpu_gemm

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROW_BLOCK = 512


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


def _check_rows(D, A_bits, B_bits, dtype, what, row0=0):
    """D (CPU torch, [rows, N]) against the oracle for rows row0.. of A."""
    rows = D.shape[0]
    for r in range(0, rows, ROW_BLOCK):
        r1 = min(rows, r + ROW_BLOCK)
        Dref, S = oracle.gemm(A_bits, B_bits, dtype, rows=(row0 + r, row0 + r1))
        assert_within_bound(D[r:r1], Dref, S, "%s rows %d..%d" % (what, row0 + r, row0 + r1 - 1))


def _dense_full(c):
    D, _ = gpu_gemm(c.A, c.B, c.out_dtype)
    assert torch.isfinite(D.float()).all()
    _check_rows(D, wl.bits(c.A), wl.bits(c.B), c.in_dtype, c.name)


def test_square_4096_every_output():
    _dense_full(wl.square_case())


def test_large_8192_every_output_in_bench_configuration():
    _dense_full(wl.large_case())


def test_fp16_large_8192_every_output():
    _dense_full(wl.large_case(dtype="fp16"))


def _grouped_device(c):
    dev = torch.device("cuda")
    return (c.A.to(dev), [b.to(dev) for b in c.Bs],
            torch.from_numpy(np.asarray(c.offsets, dtype=np.int32)).to(dev))


def _grouped_full(c):
    from blackwell_tensor_core_gb300 import ops
    A, Bs, off = _grouped_device(c)
    D = torch.full((c.total, c.N), float("nan"), dtype=c.A.dtype, device="cuda")
    ops.grouped_gemm_bf16(A.data_ptr(), [b.data_ptr() for b in Bs], D.data_ptr(), off.data_ptr(), c.G,
                          c.total, c.N, c.K, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    D = D.cpu()
    assert torch.isfinite(D.float()).all()
    A_bits = wl.bits(c.A)
    for g in range(c.G):
        r0, r1 = int(c.offsets[g]), int(c.offsets[g + 1])
        _check_rows(D[r0:r1], A_bits, wl.bits(c.Bs[g]), c.in_dtype, "%s expert %d" % (c.name, g), row0=r0)


def test_grouped_fc1_every_output():
    _grouped_full(wl.grouped_case())


def test_grouped_fc2_every_output():
    _grouped_full(wl.grouped_fc2_case())


def test_grouped_fc1_swiglu_every_output():
    from blackwell_tensor_core_gb300 import ops
    c = wl.grouped_case()
    A, Bs, off = _grouped_device(c)
    I = c.N // 2
    H = torch.full((c.total, I), float("nan"), dtype=c.A.dtype, device="cuda")
    ops.grouped_gemm_swiglu_bf16(A.data_ptr(), [b.data_ptr() for b in Bs], H.data_ptr(), off.data_ptr(),
                                 c.G, c.total, c.N, c.K, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    H = H.cpu()
    assert torch.isfinite(H.float()).all()
    A_bits = wl.bits(c.A)
    for g in range(c.G):
        r0, r1 = int(c.offsets[g]), int(c.offsets[g + 1])
        B_bits = wl.bits(c.Bs[g])
        for r in range(r0, r1, ROW_BLOCK):
            re = min(r1, r + ROW_BLOCK)
            Dref, S = oracle.gemm(A_bits, B_bits, c.in_dtype, rows=(r, re))
            Href, silu = oracle.swiglu(Dref, with_silu=True)
            W = oracle.swiglu_weight(Dref, S, silu)
            bad = oracle.bound_violations(H[r:re].double().numpy(), Href, W)
            assert not bad.any(), "expert %d rows %d..%d: %d of %d outside the SwiGLU bound" % (
                g, r, re - 1, int(bad.sum()), bad.size)

"""Helpers shared by the GPU parity tests (not collected as tests)."""
import os
from contextlib import contextmanager

import numpy as np
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl

KERNEL_ENV = {"2cta": "2cta", "1cta": "1cta", "small_m": "small_m", None: None}
OUT_TORCH = {0: torch.bfloat16, 1: torch.float32, 2: torch.float16}
OUT_NAME = {0: "bf16", 1: "fp32", 2: "fp16"}


@contextmanager
def forced_kernel(kind):
    old = os.environ.get("BWG_FORCE_KERNEL")
    if kind is None:
        os.environ.pop("BWG_FORCE_KERNEL", None)
    else:
        os.environ["BWG_FORCE_KERNEL"] = kind
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("BWG_FORCE_KERNEL", None)
        else:
            os.environ["BWG_FORCE_KERNEL"] = old


def gpu_gemm(A_cpu, B_cpu, out_dtype, kind=None, lda=None, ldb=None, ldd=None, sentinel=None):
    """Run the library on CPU-generated inputs; returns (D [M,N] CPU, full D buffer CPU)."""
    from blackwell_tensor_core_gb300 import ops
    M, K = A_cpu.shape
    N = B_cpu.shape[1]
    lda = lda or K
    ldb = ldb or N
    ldd = ldd or N
    dev = torch.device("cuda")
    Abuf = torch.zeros((M, lda), dtype=A_cpu.dtype)
    Abuf[:, :K] = A_cpu
    Bbuf = torch.zeros((K, ldb), dtype=B_cpu.dtype)
    Bbuf[:, :N] = B_cpu
    Ad = Abuf.to(dev)
    Bd = Bbuf.to(dev)
    Dd = torch.empty((M, ldd), dtype=OUT_TORCH[out_dtype], device=dev)
    Dd.fill_(float("nan") if sentinel is None else sentinel)
    fn = ops.gemm_bf16 if A_cpu.dtype == torch.bfloat16 else ops.gemm_fp16
    with forced_kernel(kind):
        fn(Ad.data_ptr(), Bd.data_ptr(), Dd.data_ptr(), M, N, K, lda, ldb, ldd, out_dtype,
           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    assert st == 0, "device error word %#x" % word
    full = Dd.cpu()
    return full[:, :N], full


def in_dtype_name(t):
    return "fp16" if t.dtype == torch.float16 else "bf16"


def assert_within_bound(D, Dref, S, what=""):
    Dv = D.double().numpy() if isinstance(D, torch.Tensor) else np.asarray(D, np.float64)
    bad = oracle.bound_violations(Dv, Dref, S)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join("(%s): got %r want %r S %r" % (tuple(i), Dv[tuple(i)], Dref[tuple(i)], S[tuple(i)])
                           for i in idx)
        raise AssertionError("%s: %d of %d outside the bound; first %s" % (what, bad.sum(), bad.size, detail))


def assert_bits_equal(D_torch, want_bits, what=""):
    got = wl.bits(D_torch.contiguous())
    if not np.array_equal(got, want_bits):
        diff = np.argwhere(got != want_bits)[:5]
        raise AssertionError("%s: %d mismatches; first at %s" % (what, int((got != want_bits).sum()),
                                                                  [tuple(d) for d in diff]))

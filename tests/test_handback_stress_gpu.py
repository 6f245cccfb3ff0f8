"""Accumulator hand-back under pressure.

The two-consumer kernels hand each TMEM accumulator back to the MMA warp with
a relaxed arrive once the epilogue's reads of it have completed, and the
dynamic scheduler releases its response slots the same way.  With K of only
two k-blocks a unit is over in a few microseconds, so hand-backs and unit
changes follow each other as fast as the kernels allow.  Integer inputs in
{-1, 0, 1} make every output exact in FP32 and in BF16 (|sum| <= 128): the
first launch must equal the oracle bit for bit, and every later launch the
first.  An accumulator overwritten before the epilogue had read it would
show up as a changed output."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl
from gpu_util import forced_kernel

pytestmark = pytest.mark.gpu

REPEATS = 60


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


def _exact(D_cpu, Dref, what):
    want = torch.from_numpy(Dref).to(torch.float64)
    bad = (D_cpu.to(torch.float64) != want).sum().item()
    assert bad == 0, "%s: %d outputs differ from the oracle" % (what, bad)


@pytest.fixture(scope="module")
def dense_case():
    M, N, K = 8192, 8192, 128  # 512 two-consumer units (or 1024 pair tiles) of 2 k-blocks
    g = wl.generator(7100)
    A = wl.randint_matrix(M, K, -1, 1, g)
    B = wl.randint_matrix(K, N, -1, 1, g)
    Dref, _ = oracle.gemm(wl.bits(A), wl.bits(B), "bf16")
    return A, B, Dref


@pytest.mark.parametrize("kind", [None, "2cta"])
@pytest.mark.parametrize("out_code", [wl.OUT_FP32, wl.OUT_BF16])
def test_dense_short_units_repeat_exactly(dense_case, kind, out_code):
    from blackwell_tensor_core_gb300 import ops
    A, B, Dref = dense_case
    (M, K), N = A.shape, B.shape[1]
    dev = torch.device("cuda")
    Ad, Bd = A.to(dev), B.to(dev)
    dt = torch.float32 if out_code == wl.OUT_FP32 else torch.bfloat16
    first = torch.full((M, N), float("nan"), dtype=dt, device=dev)
    D = torch.empty((M, N), dtype=dt, device=dev)
    h = torch.cuda.current_stream().cuda_stream
    changed = 0
    with forced_kernel(kind):
        ops.gemm_bf16(Ad.data_ptr(), Bd.data_ptr(), first.data_ptr(), M, N, K, K, N, N, out_code, h)
        for _ in range(REPEATS):
            D.fill_(float("nan"))
            ops.gemm_bf16(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, K, N, N, out_code, h)
            changed += int((D != first).sum().item())
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    _exact(first.cpu(), Dref, "first launch (%s)" % (kind or "default"))
    assert changed == 0, "%d outputs changed between repeated launches" % changed


def test_grouped_short_units_repeat_exactly():
    from blackwell_tensor_core_gb300 import ops
    counts = wl.expert_counts(4096, 8, 32, wl.generator(1005))  # the FC1 buckets
    off = wl.offsets_from_counts(counts)
    N, K = 4096, 128
    g = wl.generator(7200)
    total = int(off[-1])
    A = wl.randint_matrix(total, K, -1, 1, g)
    Bs = [wl.randint_matrix(K, N, -1, 1, g) for _ in range(len(counts))]
    dev = torch.device("cuda")
    Ad = A.to(dev)
    Bd = [b.to(dev) for b in Bs]
    offd = torch.from_numpy(np.asarray(off, dtype=np.int32)).to(dev)
    first = ops.grouped_gemm(Ad, Bd, offd)
    torch.cuda.synchronize()
    changed = 0
    D = torch.empty_like(first)
    for _ in range(REPEATS):
        D.fill_(float("nan"))
        ops.grouped_gemm(Ad, Bd, offd, out=D)
        changed += int((D != first).sum().item())
    st, word = ops.last_device_error()
    assert st == 0, hex(word)
    first = first.cpu()
    A_bits = wl.bits(A)
    for e in range(len(counts)):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        Dref, _ = oracle.gemm(A_bits, wl.bits(Bs[e]), "bf16", rows=(r0, r1))
        _exact(first[r0:r1], Dref, "expert %d" % e)
    assert changed == 0, "%d outputs changed between repeated launches" % changed

"""GPU probes of single mechanisms (cluster shared-memory exchange, TMA
128-byte swizzle, one tcgen05.mma tile read back from TMEM), each checked
against values the pages print or a plain formula, independent of the GEMM
kernels that build on them."""
import os

import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "cluster_examples.txt")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


def _golden():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split(":")
            out[k] = [int(x) for x in v.split()]
    return out


def _check(status):
    from blackwell_tensor_core_gb300 import ops
    assert status == 0, ops.status_string(status)
    torch.cuda.synchronize()
    st, word = ops.last_device_error()
    assert st == 0, hex(word)


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("n", [4, 8])
def test_cluster_pair_matches_page_examples(n):
    from blackwell_tensor_core_gb300 import ops
    gold = _golden()
    x = torch.tensor(gold["pair_sum_in"][:n], dtype=torch.float32, device="cuda")
    sums = torch.full((n,), -1.0, device="cuda")
    peers = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    _check(ops.lib().bwg_probe_cluster_pair(x.data_ptr(), sums.data_ptr(), peers.data_ptr(), n, _stream()))
    if n == 4:
        assert peers.cpu().tolist() == gold["cluster_peer_n4"]
    else:
        assert sums.cpu().tolist() == [float(v) for v in gold["pair_sum_out"]]
        assert peers.cpu().tolist() == [i ^ 1 for i in range(8)]


def test_tma_128b_swizzle_image_matches_formula():
    from blackwell_tensor_core_gb300 import ops
    src = torch.arange(64 * 64, dtype=torch.int32).to(torch.int16).view(64, 64)
    srcd = src.cuda()
    out = torch.zeros(8192, dtype=torch.uint8, device="cuda")
    _check(ops.lib().bwg_probe_tma_swizzle(srcd.data_ptr(), out.data_ptr(), _stream()))
    img = out.cpu().numpy().view(np.uint16)
    s = src.numpy().view(np.uint16)
    for r in range(64):
        for c in range(8):
            off = (r * 128 + ((c ^ (r % 8)) * 16)) // 2  # 16-bit elements
            assert np.array_equal(img[off:off + 8], s[r, 8 * c:8 * c + 8]), (r, c)


@pytest.mark.parametrize("k_steps", [1, 4])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_single_tile_mma_exact(k_steps, dtype):
    from blackwell_tensor_core_gb300 import ops
    g = wl.generator(8000 + k_steps)
    A = wl.randint_matrix(128, 64, -2, 2, g, dtype)
    B = wl.randint_matrix(64, 256, -2, 2, g, dtype)
    Ad, Bd = A.cuda(), B.cuda()  # kept alive until the probe has run
    D = torch.full((128, 256), float("nan"), dtype=torch.float32, device="cuda")
    _check(ops.lib().bwg_probe_mma(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), k_steps,
                                   1 if dtype == "fp16" else 0, _stream()))
    K = 16 * k_steps
    Dref, _ = oracle.gemm(wl.bits(A[:, :K].contiguous()), wl.bits(B[:K].contiguous()), dtype)
    assert np.array_equal(D.cpu().double().numpy(), Dref)


def _tables_by_loop(offsets, g0, G, G_total, M, n_tiles, tile_m):
    """The grouped schedule tables by their sequential definition: one group
    after the other, each row range clamped into [0, M] and after the previous
    group's end."""
    ok, tiles, prev_hi = True, 0, 0
    prefix, lo, hi = [], [], []
    for g in range(G):
        a, b = offsets[g0 + g], offsets[g0 + g + 1]
        if g0 + g == 0 and a != 0:
            ok = False
        if b < a or a < prev_hi or a < 0 or b > M:
            ok = False
        a = max(a, prev_hi)
        a = M if a > M else max(a, 0)
        b = a if b < a else min(b, M)
        prev_hi = b
        prefix.append(tiles)
        lo.append(a)
        hi.append(b)
        tiles += ((b - a + tile_m - 1) // tile_m) * n_tiles
    prefix.append(tiles)
    if g0 + G == G_total and offsets[G_total] != M:
        ok = False
    return prefix, lo, hi, ok


def test_grouped_tables_warp_matches_the_sequential_definition():
    from blackwell_tensor_core_gb300 import ops
    rng = np.random.default_rng(21)
    h = torch.cuda.current_stream().cuda_stream
    cases = []
    for G in (1, 2, 7, 31, 32, 33, 63, 64):
        counts = rng.integers(0, 1200, size=G)
        counts[rng.random(G) < 0.3] = 0
        off = [0] + [int(x) for x in np.cumsum(counts)]
        cases.append((off, 0, G, G, off[-1]))                       # valid
        bad = list(off)
        bad[G // 2] += 5000                                          # out of order, past M
        cases.append((bad, 0, G, G, off[-1]))
        neg = list(off)
        neg[0] = -3                                                  # first offset not 0
        cases.append((neg, 0, G, G, off[-1]))
        cases.append((off, 0, G, G, off[-1] + 17))                   # last != M
    long = [0] + [int(x) for x in np.cumsum(rng.integers(0, 900, size=70))]
    cases.append((long, 0, 64, 70, long[-1]))                        # first launch of 70 groups
    cases.append((long, 64, 6, 70, long[-1]))                        # second launch
    cases.append((long, 30, 40, 70, long[-1]))
    for off, g0, G, G_total, M in cases:
        for n_tiles, tile_m in ((16, 512), (3, 256)):
            d_off = torch.tensor(off, dtype=torch.int32, device="cuda")
            out = torch.full((3 * G + 2,), -7, dtype=torch.int32, device="cuda")
            _check(ops.lib().bwg_probe_grouped_tables(d_off.data_ptr(), g0, G, G_total, M, n_tiles, tile_m,
                                                      out.data_ptr(), h))
            got = out.cpu().tolist()
            prefix, lo, hi, ok = _tables_by_loop(off, g0, G, G_total, M, n_tiles, tile_m)
            assert got[:G + 1] == prefix, (g0, G, M)
            assert got[G + 1:2 * G + 1] == lo, (g0, G, M)
            assert got[2 * G + 1:3 * G + 1] == hi, (g0, G, M)
            assert got[3 * G + 1] == (1 if ok else 0), (g0, G, M)

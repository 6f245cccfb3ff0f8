"""Host-side tests of the C library (no GPU): exported symbols, argument
checks, planner values against figures printed on the pages, descriptor
encoders against words derived by hand from the PTX ISA field tables, the
128-byte swizzle, and the tile schedules."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "page_budgets.txt")


@pytest.fixture(scope="module")
def ops():
    from blackwell_tensor_core_gb300 import build as b
    b.build()
    from blackwell_tensor_core_gb300 import ops as o
    return o


def _golden():
    rows = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        rows.setdefault(key, []).append([float(v) for v in vals])
    return rows


def test_library_exports_every_declared_function(ops):
    header = open(os.path.join(ROOT, "include", "bwgemm.h"), encoding="utf-8").read()
    header = re.sub(r"/\*.*?\*/", "", header, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w ]*?[\s\*]+(\w+)\s*\(", header, flags=re.M)
    names = [n for n in names if n not in ("if", "return")]
    assert {"gemm_bf16", "gemm_fp16", "grouped_gemm_bf16", "grouped_gemm_swiglu_bf16",
            "grouped_gemm_swiglu_fp16", "bwg_last_device_error"} <= set(names)
    raw = ctypes.CDLL(ops.LIB_PATH)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing


def test_swiglu_argument_checks_need_no_device(ops):
    """Host-side checks of the SwiGLU entry point run before any CUDA call:
    the up block must start on a 16-byte boundary (N a multiple of 16)."""
    L = ops.lib()
    arr = (ctypes.c_void_p * 1)(ctypes.c_void_p(256))
    Bp = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    assert L.grouped_gemm_swiglu_bf16(256, Bp, 256, 256, 1, 8, 24, 64, None) == 2
    assert L.grouped_gemm_swiglu_fp16(256, Bp, 256, 256, 1, 8, 40, 64, None) == 2
    assert L.grouped_gemm_swiglu_bf16(256, Bp, 256, 256, -1, 8, 32, 64, None) == 1
    assert L.grouped_gemm_swiglu_bf16(256, Bp, 264, 256, 1, 8, 32, 64, None) == 2  # H misaligned
    assert L.grouped_gemm_swiglu_bf16(256, Bp, 256, 256, 0, 8, 32, 64, None) == 0  # nothing to do


def test_dynamic_schedule_plan(ops, monkeypatch):
    """BWG_SCHED=clc: the two-consumer plan launches one pair per unit; the
    last-wave cut is still computed for the pairs that run at once."""
    static = ops.plan(8192, 8192, 8192, force_kernel=ops.KERNEL_2CTA_2C)
    assert static.dynamic == 0 and static.workers == 76 and static.grid == 152
    monkeypatch.setenv("BWG_SCHED", "clc")
    dyn = ops.plan(8192, 8192, 8192, force_kernel=ops.KERNEL_2CTA_2C)
    assert dyn.dynamic == 1 and dyn.workers == 76
    assert dyn.units == static.units and dyn.grid == 2 * dyn.units
    # other kernels keep the static schedule
    assert ops.plan(8192, 8192, 8192, force_kernel=ops.KERNEL_2CTA).dynamic == 0


def test_streamk_last_wave_plan(ops, monkeypatch):
    """Stream-K of the last wave (opt-in): taken for 4096^3 (52 of 128 tiles)
    and 8192^3 (56 of 512), not when the tiles fill whole waves, not for K
    below 4 k-blocks; the per-pair segment bound covers every pair's range."""
    assert ops.plan(4096, 4096, 4096).streamk == 0  # off by default
    monkeypatch.setenv("BWG_STREAMK_DENSE", "1")
    p = ops.plan(4096, 4096, 4096)
    assert (p.kernel, p.streamk, p.sk_tiles, p.workers) == (ops.KERNEL_2CTA_2C, 1, 52, 76)
    assert p.units == p.sk_segs * 76 + 128 - 52
    assert ops.plan(8192, 8192, 8192).sk_tiles == 56
    assert ops.plan(4096, 4096, 64).streamk == 0
    assert ops.plan(512 * 76 // 4, 1024, 4096).sk_tiles == 0  # 76 tiles: whole waves
    monkeypatch.setenv("BWG_STREAMK_DENSE", "0")
    assert ops.plan(4096, 4096, 4096).streamk == 0
    L = ops.lib()
    for T, C, kb in [(128, 76, 64), (512, 76, 128), (95, 76, 8), (8, 76, 64), (10, 3, 7)]:
        segs = ctypes.c_int(0)
        R = L.bwg_streamk_tiles(T, C, kb, 1 << 30, ctypes.byref(segs))
        assert R == T % C
        W = R * kb
        for w in range(C):
            lo, hi = W * w // C, W * (w + 1) // C
            pos, n = lo, 0
            while pos < hi:
                pos = min((pos // kb + 1) * kb, hi)
                n += 1
            assert n <= segs.value, (T, C, kb, w)


def test_status_strings(ops):
    assert ops.status_string(0) == "ok"
    assert "align" in ops.status_string(2)
    assert ops.lib().bwg_version().decode().startswith("bwgemm")


def test_argument_checks(ops):
    ok, inv, ali = 0, 1, 2
    A, B, D = 0x10000, 0x20000, 0x30000
    c = ops.check_gemm_args
    assert c(A, B, D, 256, 256, 512, 512, 256, 256, 0) == ok
    assert c(A, B, D, 256, 256, 512, 512, 256, 256, 7) == inv          # bad out dtype
    assert c(A, B, D, -1, 256, 512, 512, 256, 256, 0) == inv
    assert c(0, B, D, 256, 256, 512, 512, 256, 256, 0) == inv          # null A
    assert c(A, B, 0, 256, 256, 512, 512, 256, 256, 0) == inv          # null D
    assert c(A, B, D, 256, 256, 512, 500, 256, 256, 0) == inv          # lda < K
    assert c(A, B, D, 256, 256, 512, 512, 200, 256, 0) == inv          # ldb < N
    assert c(A, B, D, 256, 256, 512, 512, 256, 100, 0) == inv          # ldd < N
    assert c(A + 8, B, D, 256, 256, 512, 512, 256, 256, 0) == ali      # misaligned A
    assert c(A, B, D, 256, 256, 512, 516, 256, 256, 0) == ali          # lda*2 not 16-byte
    assert c(A, B, D, 256, 260, 512, 512, 260, 264, 0) == ali          # ldb*2 = 520
    assert c(A, B, D, 256, 260, 512, 512, 264, 260, 1) == ok           # fp32 D: 260*4 = 1040
    assert c(A, B, D, 256, 260, 512, 512, 264, 260, 0) == ali          # bf16 D: 520
    assert c(0, 0, 0, 0, 256, 512, 0, 0, 0, 0) == ok                   # empty problem
    assert c(0, 0, D, 4, 8, 0, 0, 0, 8, 0) == ok                       # K = 0: only D needed


def test_planner_matches_page_calculator(ops):
    g = _golden()
    M, N, K, stages, tiles, cov, kib, kblocks = g["calculator"][0]
    p = ops.plan(int(M), int(N), int(K), force_kernel=ops.KERNEL_2CTA, force_stages=int(stages))
    assert (p.tile_m, p.tile_n, p.tile_k) == (256, 256, 64)
    assert p.tiles == tiles
    assert round(p.coverage * 100, 1) == cov
    assert p.smem_input_per_cta // 1024 == kib
    assert p.k_blocks == kblocks


def test_planner_stage_and_barrier_accounting(ops):
    g = _golden()
    lone, pair = g["per_cta_kib"][0]
    p1 = ops.plan(512, 512, 512, force_kernel=ops.KERNEL_1CTA, force_stages=2)
    p2 = ops.plan(512, 512, 512, force_kernel=ops.KERNEL_2CTA, force_stages=2)
    assert p1.smem_input_per_cta // 2 // 1024 == lone
    assert p2.smem_input_per_cta // 2 // 1024 == pair
    assert 2 * 256 * 256 * 64 == g["round_flops"][0][0]
    assert p2.smem_input_per_cta // 2 // 1024 == g["stage_kib"][0][0]
    staging_kib = 32  # four epilogue warps x two 4 KiB boxes
    for depth, total in g["depth_total_kib"]:
        p = ops.plan(4096, 4096, 4096, force_kernel=ops.KERNEL_2CTA, force_stages=int(depth))
        assert p.smem_input_per_cta // 1024 + staging_kib == total
        assert p.smem_total <= 232448
    assert p2.tx_bytes == g["tx_bytes"][0][0]
    assert 128 * 256 * 4 // 1024 == g["accumulator_kib"][0][0]


def test_planner_choices(ops):
    big = ops.plan(8192, 8192, 8192)
    assert big.kernel == ops.KERNEL_2CTA_2C and big.stages == 4 and big.tiles == 512
    assert big.tile_m == 512 and big.grid == 152 and big.smem_total <= 232448
    assert ops.plan(2048, 2048, 2048).kernel == ops.KERNEL_2CTA  # 32 big tiles < 76 pairs
    small = ops.plan(72, 16384, 7168)
    assert small.kernel == ops.KERNEL_SMALL_M and small.mma_n == 80
    # whole 128-column tiles walking K in step; stream-K for few or too many tiles
    assert small.tile_n == 128 and small.tiles == 128 and small.streamk == 0 and small.grid == 128
    assert ops.plan(72, 24576, 7168).streamk == 1 and ops.plan(72, 19456, 7168).streamk == 0
    assert small.split == 1
    assert small.smem_total <= 232448 and small.stages >= 4
    for tokens, n in _golden()["n_compute"]:
        assert ops.plan(int(tokens), 4096, 4096).mma_n == n
    assert ops.plan(0, 10, 10).kernel == ops.KERNEL_NONE
    assert ops.plan(10, 10, 0).kernel == ops.KERNEL_ZERO
    assert ops.plan(129, 10, 10).kernel == ops.KERNEL_2CTA
    p2 = ops.plan(512, 512, 512, force_kernel=ops.KERNEL_2CTA_2C, force_stages=2)
    assert p2.smem_input_per_cta // 2 == 48 * 1024  # two A blocks + one B block per CTA per stage
    assert p2.tx_bytes == 2 * 48 * 1024
    assert ops.plan(128, 10, 10).kernel == ops.KERNEL_SMALL_M


def test_small_m_cluster_split_plan(ops, monkeypatch):
    """Few column tiles (at most half the SMs): a cluster of F CTAs shares
    each tile's k-blocks, F chosen to keep the most SMs streaming with every
    cluster co-resident (host estimate: 76, 36, 15 clusters of 2, 4, 8 on 152
    SMs) and at least two k-blocks per CTA."""
    cases = {(72, 4096, 7168): 4, (72, 8192, 7168): 2, (72, 7168, 2048): 2, (72, 1000, 4096): 8,
             (16, 2048, 4096): 4, (128, 4104, 640): 4, (72, 16384, 7168): 1, (72, 256, 64): 1,
             (72, 24576, 7168): 1, (72, 1000, 448): 2}
    for shape, F in cases.items():
        p = ops.plan(*shape)
        assert p.split == F, (shape, p.split)
        if F > 1:
            assert p.streamk == 0 and p.grid == p.tiles * F and p.k_blocks >= 2 * F
    monkeypatch.setenv("BWG_SMALL_M_SPLIT", "0")
    assert ops.plan(72, 4096, 7168).split == 1 and ops.plan(72, 4096, 7168).streamk == 1
    monkeypatch.setenv("BWG_SMALL_M_SPLIT", "2")
    assert ops.plan(72, 4096, 7168).split == 2
    monkeypatch.delenv("BWG_SMALL_M_SPLIT")
    monkeypatch.setenv("BWG_STREAMK", "1")
    assert ops.plan(72, 4096, 7168).split == 1 and ops.plan(72, 4096, 7168).streamk == 1


def test_small_m_load_grouping_plan(ops, monkeypatch):
    """How the small-M kernel fills its ring: one load of B^T a stage when the
    3-D channel-group view tiles B (N a multiple of 64), else two; two stages
    a load of B^T and of A when K (and N) are multiples of 64."""
    cases = {(72, 16384, 7168): (1, 1), (72, 4096, 7168): (1, 1), (100, 1000, 640): (2, 0),
             (33, 312, 1016): (2, 0), (72, 16384, 1000): (1, 0), (16, 2048, 4096): (1, 1),
             (128, 4104, 640): (2, 0), (128, 4096, 640): (1, 1), (72, 1000, 448): (2, 0)}
    for shape, (bt, pair) in cases.items():
        p = ops.plan(*shape)
        assert p.kernel == ops.KERNEL_SMALL_M and (p.bt_loads, p.pair_loads) == (bt, pair), shape
    assert ops.plan(128, 4096, 640).stages == 7  # odd ring: the last stage is filled alone
    assert ops.plan(256, 256, 256).pair_loads == 0  # not the small-M kernel
    # the channel-group view needs every tile to start on a group of 64
    for tile_n, want in ((64, (1, 1)), (80, (2, 0)), (112, (2, 0)), (128, (1, 1))):
        monkeypatch.setenv("BWG_SMALL_M_TILE_N", str(tile_n))
        p = ops.plan(72, 1024, 640)
        assert p.tile_n == tile_n and (p.bt_loads, p.pair_loads) == want, tile_n
    monkeypatch.delenv("BWG_SMALL_M_TILE_N")
    monkeypatch.setenv("BWG_SMALL_M_PAIRS", "0")
    assert ops.plan(72, 16384, 7168).pair_loads == 0 and ops.plan(72, 16384, 7168).bt_loads == 1


def test_instruction_descriptor_words(ops):
    # Fields (PTX ISA, tcgen05 instruction descriptor for kind::f16):
    # bit 4 = D is F32, bits 7-9 A format (1 = BF16), bits 10-12 B format,
    # bit 15/16 A/B MN-major, bits 17-22 N>>3, bits 24-28 M>>4.
    # Pair tile, BF16, A K-major, B MN-major, M = N = 256:
    want = (1 << 4) | (1 << 7) | (1 << 10) | (1 << 16) | ((256 >> 3) << 17) | ((256 >> 4) << 24)
    assert want == 0x10410490
    assert ops.lib().bwg_idesc_f16(1, 0, 1, 256, 256) == want
    # swapped small-M kernel, FP16, A MN-major, B K-major, M = 128, N = 80
    want = (1 << 4) | (1 << 15) | ((80 >> 3) << 17) | ((128 >> 4) << 24)
    assert ops.lib().bwg_idesc_f16(0, 1, 0, 128, 80) == want
    # the N field alone, as the MegaMoE page prints it: (N >> 3) << 17
    for n in range(16, 257, 16):
        w = ops.lib().bwg_idesc_f16(1, 0, 0, 128, n)
        assert (w >> 17) & 0x3F == n >> 3
        assert w & ~(0x3F << 17) == ops.lib().bwg_idesc_f16(1, 0, 0, 128, 16) & ~(0x3F << 17)


def test_shared_memory_descriptor_words(ops):
    # start >> 4 in bits 0-13, LBO >> 4 in 16-29, SBO >> 4 in 32-45,
    # version 1 at bit 46, swizzle mode in 61-63 (2 = 128-byte).
    d = ops.lib().bwg_smem_desc(0x1400, 8192, 1024, 2)
    assert d == (0x140) | (512 << 16) | (64 << 32) | (1 << 46) | (2 << 61)
    d = ops.lib().bwg_smem_desc(0x3FFF0, 16, 1024, 2)
    assert d & 0x3FFF == 0x3FFF
    assert (d >> 16) & 0x3FFF == 1


def test_swizzle_matches_page_formula_and_is_a_permutation(ops):
    f = ops.lib().bwg_swizzle128_offset
    for row in range(64):
        offs = [f(row, c) for c in range(8)]
        # "GEMM优化（三）" 2.1: physical = row*128 + ((chunk ^ (row % 8)) * 16)
        assert offs == [row * 128 + ((c ^ (row % 8)) * 16) for c in range(8)]
        assert sorted(offs) == [row * 128 + 16 * c for c in range(8)]
    # the eight rows of one atom put a given chunk in eight different bank groups
    for c in range(8):
        assert len({(f(r, c) % 128) // 16 for r in range(8)}) == 8


@pytest.mark.parametrize("mt,nt,gm", [(32, 32, 8), (16, 16, 8), (5, 7, 8), (9, 3, 4), (1, 1, 8), (13, 11, 16)])
def test_raster_order_covers_every_tile_once(ops, mt, nt, gm):
    m = ctypes.c_int()
    n = ctypes.c_int()
    seen = set()
    for t in range(mt * nt):
        ops.lib().bwg_raster_tile(t, mt, nt, gm, ctypes.byref(m), ctypes.byref(n))
        assert 0 <= m.value < mt and 0 <= n.value < nt
        seen.add((m.value, n.value))
        # inside one raster group the row index stays within the group's rows
        assert m.value // gm == t // (gm * nt)
    assert len(seen) == mt * nt


def _schedule(ops, offsets, N, tile_m):
    G = len(offsets) - 1
    ia = ctypes.c_int * (G + 1)
    off = ia(*offsets)
    prefix, lo, hi = ia(), ia(), ia()
    ok = ops.lib().bwg_grouped_schedule(off, G, offsets[-1], N, tile_m, prefix, lo, hi)
    return ok, list(prefix), list(lo)[:G], list(hi)[:G]


def test_grouped_schedule_covers_every_row_and_column_once(ops):
    counts = [300, 0, 256, 1, 0, 511, 1024, 0]
    offsets = [0] + list(np.cumsum(counts))
    N, tile_m = 600, 256
    ok, prefix, lo, hi = _schedule(ops, offsets, N, tile_m)
    assert ok == 1
    n_tiles = (N + 255) // 256
    want = [((c + tile_m - 1) // tile_m) * n_tiles for c in counts]
    assert prefix == list(np.concatenate([[0], np.cumsum(want)]))
    G = len(counts)
    covered = np.zeros((offsets[-1], n_tiles), dtype=int)
    g, m0, n0, re_ = (ctypes.c_int() for _ in range(4))
    P = (ctypes.c_int * (G + 1))(*prefix)
    L = (ctypes.c_int * G)(*lo)
    H = (ctypes.c_int * G)(*hi)
    for t in range(prefix[-1]):
        ops.lib().bwg_grouped_tile(t, G, P, L, H, tile_m, ctypes.byref(g), ctypes.byref(m0),
                                   ctypes.byref(n0), ctypes.byref(re_))
        assert counts[g.value] > 0
        assert offsets[g.value] <= m0.value < offsets[g.value + 1] == re_.value
        rows = range(m0.value, min(m0.value + tile_m, re_.value))
        covered[list(rows), n0.value // 256] += 1
    assert (covered == 1).all()


def test_grouped_tile_group_lookup_matches_a_scan(ops):
    # The device finds a unit's group by bisection over the prefix of tiles
    # per group; it must agree with a plain scan, also with runs of empty
    # groups at the start, in the middle and at the end.
    rng = np.random.default_rng(11)
    N, tile_m = 512, 512
    n_tiles = 2
    for trial in range(40):
        G = int(rng.integers(1, 65))
        counts = rng.integers(0, 1500, size=G)
        counts[rng.random(G) < 0.3] = 0
        offsets = [0] + [int(x) for x in np.cumsum(counts)]
        ok, prefix, lo, hi = _schedule(ops, offsets, N, tile_m)
        assert ok == 1
        P = (ctypes.c_int * (G + 1))(*prefix)
        L = (ctypes.c_int * G)(*lo)
        H = (ctypes.c_int * G)(*hi)
        g, m0, n0, re_ = (ctypes.c_int() for _ in range(4))
        for t in range(prefix[-1]):
            ops.lib().bwg_grouped_tile(t, G, P, L, H, tile_m, ctypes.byref(g), ctypes.byref(m0),
                                       ctypes.byref(n0), ctypes.byref(re_))
            want = 0
            while want + 1 < G and prefix[want + 1] <= t:
                want += 1
            assert g.value == want, (trial, t)
            assert counts[want] > 0


def test_grouped_schedule_flags_bad_offsets(ops):
    assert _schedule(ops, [0, 10, 5, 20], 256, 256)[0] == 0      # decreasing
    assert _schedule(ops, [3, 10, 20], 256, 256)[0] == 0         # first != 0
    ok, prefix, lo, hi = _schedule(ops, [0, 10, 5, 20], 256, 256)
    assert all(l <= h for l, h in zip(lo, hi)) and lo[1] >= hi[0]  # clamped, disjoint


@pytest.mark.parametrize("T,C", [(1024, 76), (256, 76), (1, 76), (76, 76), (77, 76), (114, 76),
                                 (115, 76), (2048, 152), (5, 4), (40, 76)])
def test_last_wave_split_covers_every_column_once(ops, T, C):
    R = ops.lib().bwg_tail_split(T, C)
    rem = T % C
    # halves cost 0.75 of a tile: worth it while they fit in one wave
    assert R == (rem if 0 < rem and 2 * rem <= C else 0)
    units = T + R
    tile, off, width = (ctypes.c_int() for _ in range(3))
    cover = {}
    last_wave = (units - 1) // C
    for u in range(units):
        ops.lib().bwg_unit_tile(u, T, R, 256, ctypes.byref(tile), ctypes.byref(off), ctypes.byref(width))
        assert width.value in (256, 128)
        if width.value == 128:
            assert u // C == last_wave  # split units all run in the last wave
        for c in range(off.value, off.value + width.value, 64):
            cover[(tile.value, c)] = cover.get((tile.value, c), 0) + 1
    assert sorted(cover) == [(t, c) for t in range(T) for c in range(0, 256, 64)]
    assert set(cover.values()) == {1}
    # the split never lengthens the schedule and shortens it whenever it applies
    waves_before = -(-T // C)
    waves_after = ((T - R) // C + 0.5) if R else waves_before  # in whole-tile times
    assert waves_after <= waves_before
    if R:
        assert waves_after == waves_before - 0.5


def test_plan_reports_split_units(ops):
    big = ops.plan(8192, 8192, 8192, force_kernel=ops.KERNEL_2CTA)
    assert big.tiles == 1024 and big.units == 1024 + 1024 % 76
    mid = ops.plan(4096, 4096, 4096, force_kernel=ops.KERNEL_2CTA)
    assert mid.units == 256 + 256 % 76
    two = ops.plan(8192, 8192, 8192)
    # remainder 56 of 76: quarters (3 x 0.5) and halves (2 x 0.833) both lose to 1.0
    assert two.tiles == 512 and two.sk_tiles == 0 and two.units == 512
    assert ops.plan(2048, 5120, 128).units == 80 - 4 + 4 * 4       # 4 left over: quarters
    assert ops.plan(1024, 13568, 64).units == 106 - 30 + 2 * 30    # 30 left over: halves


@pytest.mark.parametrize("tiles,kb,C", [(128, 112, 152), (128, 112, 128), (3, 1, 152), (1, 200, 152),
                                        (10, 7, 4), (300, 16, 152), (128, 2, 152)])
def test_streamk_ranges_cover_each_tile_iteration_once(ops, tiles, kb, C):
    L = ops.lib()
    W = tiles * kb
    begins = [L.bwg_streamk_begin(i, W, C) for i in range(C + 1)]
    assert begins[0] == 0 and begins[-1] == W
    assert all(b <= c for b, c in zip(begins, begins[1:]))
    sizes = [c - b for b, c in zip(begins, begins[1:])]
    assert max(sizes) - min(sizes) <= 1  # even shares
    first, count = ctypes.c_int(), ctypes.c_int()
    for t in range(tiles):
        L.bwg_streamk_tile_workers(t, kb, W, C, ctypes.byref(first), ctypes.byref(count))
        owners = sorted({i for i in range(C) for p in range(begins[i], begins[i + 1]) if t * kb <= p < (t + 1) * kb})
        assert owners == list(range(first.value, first.value + count.value))


def test_grouped_swapped_tiles_are_the_short_group_ends(ops):
    L = ops.lib()
    assert L.bwg_grouped_swap_rows(1024, 1030, 256) == 6      # 6-row tail: swapped
    assert L.bwg_grouped_swap_rows(1024, 1152, 256) == 128    # 128 rows: swapped
    assert L.bwg_grouped_swap_rows(1024, 1153, 256) == 0      # 129 rows: padded tile
    assert L.bwg_grouped_swap_rows(0, 2048, 256) == 0         # full tile
    assert L.bwg_grouped_swap_rows(0, 37, 256) == 37          # whole small group
    # the expert counts of the FC1 workload: which tails go swapped
    from blackwell_tensor_core_gb300 import workloads as wl
    counts = wl.expert_counts(4096, 8, 32, wl.generator(1005))
    swapped = [c % 256 for c in counts if 0 < c % 256 <= 128]
    assert len(swapped) == 15 and max(swapped) == 68


@pytest.mark.parametrize("T,C", [(512, 76), (128, 76), (16, 76), (1024, 76), (90, 76), (3, 2), (80, 76),
                                 (106, 76)])
def test_quarter_split_for_two_consumer_tiles(ops, T, C):
    L = ops.lib()
    f = ctypes.c_int()
    R = L.bwg_tail_split_f(T, C, 4, ctypes.byref(f))
    rem = T % C
    if rem == 0:
        assert R == 0
        return
    # the chosen cut gives the cheapest last wave, preferring fewer parts
    cost = {1: 1000, 2: 833, 4: 500}
    best = min((-(-k * rem // C) * cost[k], k) for k in (1, 2, 4))
    if best[1] == 1:
        assert R == 0
    else:
        assert R == rem and f.value == best[1]
    units = T - R + R * max(f.value, 1)
    tile, part, parts = (ctypes.c_int() for _ in range(3))
    seen = {}
    for u in range(units):
        L.bwg_unit_part(u, T, R, f.value, ctypes.byref(tile), ctypes.byref(part), ctypes.byref(parts))
        if parts.value > 1:
            assert u >= T - R  # parts of cut tiles come after every whole tile
        seen.setdefault(tile.value, []).append((part.value, parts.value))
    for t in range(T):
        got = sorted(seen[t])
        n = got[0][1]
        assert got == [(k, n) for k in range(n)]


def test_gemm_binding_rejects_bad_tensors_before_any_call(ops):
    """The torch-level wrapper checks shapes and dtypes on the host, so a
    wrong output buffer never reaches the kernels (an `out` with fewer rows
    than M would otherwise be written past its end)."""
    import torch
    A = torch.zeros((72, 64), dtype=torch.bfloat16)
    B = torch.zeros((64, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match=r"out must be \[72, 128\]"):
        ops.gemm(A, B, out=torch.zeros((71, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match=r"out must be \[72, 128\]"):
        ops.gemm(A, B, out=torch.zeros((72, 120), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="inner dimensions"):
        ops.gemm(A, torch.zeros((65, 128), dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        ops.gemm(A, B.to(torch.float16))
    with pytest.raises(TypeError):
        ops.gemm(A, B, out=torch.zeros((72, 128), dtype=torch.float64))
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops.gemm(A, B)  # host tensors: the library works on device memory only


def test_host_buffer_binding_checks_shapes_and_buffers(ops):
    """gemm_bf16_host takes raw pointers; its wrapper checks the host
    tensors' shapes and dtypes and that the device buffers are CUDA buffers
    large enough for A, B and D before calling it."""
    import torch
    hA = torch.zeros((64, 32), dtype=torch.bfloat16)
    hB = torch.zeros((32, 48), dtype=torch.bfloat16)
    hD = torch.zeros((64, 48), dtype=torch.bfloat16)
    dev = [torch.zeros(1, dtype=torch.uint8)] * 3
    with pytest.raises(ValueError, match="shapes must be"):
        ops.gemm_bf16_host(hA, hB, torch.zeros((64, 40), dtype=torch.bfloat16), *dev)
    with pytest.raises(ValueError, match="shapes must be"):
        ops.gemm_bf16_host(hA, torch.zeros((33, 48), dtype=torch.bfloat16), hD, *dev)
    with pytest.raises(TypeError):
        ops.gemm_bf16_host(hA.half(), hB, hD, *dev)
    with pytest.raises(ValueError, match="dense host tensor"):
        ops.gemm_bf16_host(hA.t().contiguous().t(), hB, hD, *dev)
    with pytest.raises(ValueError, match="dA must be a dense CUDA buffer of at least 4096 bytes"):
        ops.gemm_bf16_host(hA, hB, hD, *dev)


def test_every_planner_override_is_documented_in_the_header():
    """Each BWG_* environment variable the library reads is listed in the
    public header's planner-override block."""
    import re
    csrc = os.path.join(ROOT, "blackwell_tensor_core_gb300", "csrc")
    read = set()
    for name in os.listdir(csrc):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                read |= set(re.findall(r'getenv\("(BWG_[A-Z0-9_]+)"\)', f.read()))
    with open(os.path.join(ROOT, "include", "bwgemm.h"), encoding="utf-8") as f:
        header = f.read()
    block = header[header.index("Planner overrides"):]
    block = block[:block.index("*/")]
    listed = set(re.findall(r"\*\s+(BWG_[A-Z0-9_]+)\s", block))
    assert read, "no overrides found"
    assert read <= listed, "undocumented: %s" % sorted(read - listed)

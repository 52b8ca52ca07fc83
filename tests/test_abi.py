"""CPU-side checks of the C ABI: the library loads and exports every declared symbol, and
the host logic (argument validation, tile scheduler, wave model, planner) behaves as the
lecture pages' figures require.  No test here launches a kernel."""
import ctypes
import glob
import os
import re

import pytest

import tensor_core_tiled_gb300 as tct
from tests.golden import figures

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names.update(re.findall(r"TCT_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol(tct_lib):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert declared == set(tct.EXPORTED)
    for name in declared:
        assert hasattr(tct_lib, name), name
        assert ctypes.cast(getattr(tct_lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(tct_lib):
    assert "sm_103a" in tct.version()
    for code in range(5):
        assert tct.status_string(code)
    assert tct.status_string(99) == "unknown status"


def test_invalid_arguments_rejected_before_any_device_work(tct_lib):
    p = 1 << 20  # never dereferenced: validation fails first
    bad = [
        (p, p, p, -1, 4, 4, 4, 4, 4),      # negative M
        (p, p, p, 4, 4, 4, 3, 4, 4),       # lda < K
        (p, p, p, 4, 4, 4, 4, 3, 4),       # ldb < N
        (p, p, p, 4, 4, 4, 4, 4, 3),       # ldc < N
        (0, p, p, 4, 4, 4, 4, 4, 4),       # NULL A
        (p, 0, p, 4, 4, 4, 4, 4, 4),       # NULL B
        (p, p, 0, 4, 4, 4, 4, 4, 4),       # NULL C
        (p + 1, p, p, 4, 4, 4, 4, 4, 4),   # A not FP16-aligned
        (p, p, p + 2, 4, 4, 4, 4, 4, 4),   # C not FP32-aligned
        (p, p, p, 1 << 31, 4, 4, 4, 4, 4),  # M too large
    ]
    for args in bad:
        assert tct.gemm_f16_f32(*args, 0) == tct.GEMM_ERR_INVALID_ARG, args
        assert tct.gemm_f16_f32_host(*args, 0) == tct.GEMM_ERR_INVALID_ARG, args
    assert tct.gemm_f16_f32_host(0, 0, 0, 0, 5, 7, 7, 5, 5, 0) == tct.GEMM_OK
    for fn in (tct.softmax_rows_f32, tct.softmax_rows_f32_host):
        assert fn(p, p, -1, 4, 4, 4, 0) == tct.GEMM_ERR_INVALID_ARG
        assert fn(p, p, 4, 8, 7, 8, 0) == tct.GEMM_ERR_INVALID_ARG      # ldx < N
        assert fn(p, p, 4, 8, 8, 12, 0) == tct.GEMM_ERR_INVALID_ARG     # in place, ldx != ldy
        assert fn(p + 2, p + 64, 4, 8, 8, 8, 0) == tct.GEMM_ERR_INVALID_ARG
        assert fn(0, p, 4, 8, 8, 8, 0) == tct.GEMM_ERR_INVALID_ARG
        assert fn(0, 0, 0, 8, 8, 8, 0) == tct.GEMM_OK
    # more output tiles than the kernel's 32-bit tile index: rejected by the planner
    huge = (1 << 31) - 1
    with pytest.raises(tct.GemmError):
        tct.gemm_f16_f32_plan(huge, huge, 64, num_sms=152)
    assert tct.load().gemm_f16_f32_plan(huge, huge, 64, 64, huge, 152, None,
                                        ctypes.byref(tct.GemmPlan())) == tct.GEMM_ERR_INVALID_ARG
    # empty output is a no-op that needs no device
    assert tct.gemm_f16_f32(0, 0, 0, 0, 5, 7, 7, 5, 5, 0) == tct.GEMM_OK
    assert tct.gemm_f16_f32(0, 0, 0, 5, 0, 7, 7, 0, 0, 0) == tct.GEMM_OK
    # bad options
    assert tct.gemm_f16_f32_ex(p, p, p, 4, 4, 4, 4, 4, 4, 0, tile_n=96) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_f16_f32_ex(p, p, p, 4, 4, 4, 4, 4, 4, 0, stages=9) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_f16_f32_ex(p, p, p, 4, 4, 4, 4, 4, 4, 0, group_m=-1) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_f16_f32_ex(p, p, p, 4, 4, 4, 4, 4, 4, 0, cta_group=3) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_f16_f32_ex(p, p, p, 4, 4, 4, 4, 4, 4, 0, stream_k=4) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_f16_f32_ex(p, p, p, 4, 4, 4, 4, 4, 4, 0, fault_inject=4) == tct.GEMM_ERR_INVALID_ARG
    # generalised entry: bad type or op, and leading dimensions checked against the storage
    assert tct.gemm_f32acc(2, 0, 0, p, p, p, 4, 4, 4, 4, 4, 4, 0) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_f32acc(0, 2, 0, p, p, p, 4, 4, 4, 4, 4, 4, 0) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_f32acc(1, 1, 0, p, p, p, 8, 4, 2, 4, 4, 4, 0) == tct.GEMM_ERR_INVALID_ARG   # lda < M
    assert tct.gemm_f32acc(1, 0, 1, p, p, p, 4, 8, 6, 6, 4, 8, 0) == tct.GEMM_ERR_INVALID_ARG   # ldb < K
    assert tct.gemm_f32acc(1, 1, 1, 0, 0, 0, 0, 4, 4, 1, 4, 4, 0) == tct.GEMM_OK                # empty
    # epilogue entry: bad C type, misaligned typed C or bias, non-finite scale
    assert tct.gemm_ex(0, 0, 0, p, p, p, 3, 4, 4, 4, 4, 4, 4) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_ex(0, 0, 0, p, p, p + 2, 2, 4, 4, 4, 4, 4, 4) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_ex(0, 0, 0, p, p, p + 1, 0, 4, 4, 4, 4, 4, 4) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_ex(0, 0, 0, p, p, p, 2, 4, 4, 4, 4, 4, 4, bias=p + 2, bias_type=2) == tct.GEMM_ERR_INVALID_ARG
    assert tct.gemm_ex(0, 0, 0, p, p, p, 2, 4, 4, 4, 4, 4, 4, alpha=float("inf")) == tct.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("num_m,num_n", [(9, 9), (7, 14), (32, 16), (13, 5), (1, 40), (40, 1)])
@pytest.mark.parametrize("group_m", [1, 2, 3, 4, 8, 16])
def test_tile_order_is_a_bijection(tct_lib, num_m, num_n, group_m):
    seen = set()
    for t in range(num_m * num_n):
        m, n = tct.gemm_tile_coord(t, num_m, num_n, group_m)
        assert 0 <= m < num_m and 0 <= n < num_n
        seen.add((m, n))
    assert len(seen) == num_m * num_n


def test_tile_order_row_major_and_grouped(tct_lib):
    # group_m = 1 is row-major
    assert [tct.gemm_tile_coord(t, 3, 4, 1) for t in range(5)] == [(0, 0), (0, 1), (0, 2), (0, 3), (1, 0)]
    # inside a group the index walks down the rows first
    assert [tct.gemm_tile_coord(t, 9, 9, 3) for t in range(4)] == [(0, 0), (1, 0), (2, 0), (0, 1)]
    # the last group may be shorter than group_m
    assert tct.gemm_tile_coord(9 * 8, 9, 9, 4) == (8, 0)
    assert tct.gemm_tile_coord(9 * 8 + 1, 9, 9, 4) == (8, 1)


def test_page_grouping_example_90_vs_54(tct_lib):
    """9x9 output blocks, K = 9 blocks: the first 9 programs read 90 blocks in row-major
    order and 54 with GROUP_M = 3 ("06_triton_style.py" demo 2)."""
    fig = figures.load()

    def blocks_read(group_m):
        coords = [tct.gemm_tile_coord(t, 9, 9, group_m) for t in range(9)]
        rows = {m for m, _ in coords}
        cols = {n for _, n in coords}
        return len(rows) * 9 + len(cols) * 9

    assert blocks_read(1) == fig["group9_rowmajor_blocks"]
    assert blocks_read(3) == fig["group9_grouped3_blocks"]


def test_page_wave_quantisation_example(tct_lib):
    """A100, 108 SMs, 256x128 tiles: n = 1792 -> 98 tiles in 1 wave, n = 1793 -> 120 tiles in
    2 waves ("02_gpu_execution_model.py" part 5)."""
    fig = figures.load()
    sms = int(fig["wave_sms"])
    t, w, u = tct.gemm_wave_model(1792, 1792, 256, 128, sms)
    assert (t, w) == (fig["wave_1792_tiles"], fig["wave_1792_waves"])
    assert u == pytest.approx(98 / 108)
    t, w, u = tct.gemm_wave_model(1793, 1793, 256, 128, sms)
    assert (t, w) == (fig["wave_1793_tiles"], fig["wave_1793_waves"])
    assert u == pytest.approx(120 / 216)
    with pytest.raises(tct.GemmError):
        tct.gemm_wave_model(0, 5, 128, 128, 10)


def test_planner_on_gb300_shapes(tct_lib):
    sms = 152
    p = tct.gemm_f16_f32_plan(8192, 8192, 8192, num_sms=sms)
    # the CTA-pair 256x256 tile: 32 x 32 tiles over 76 pairs, 13 whole waves, the last 36
    # tiles each split into two k-halves on 72 of the 76 pairs
    assert (p["cta_group"], p["tile_m"], p["tile_n"], p["tile_k"]) == (2, 256, 256, 64)
    assert p["grid"] == sms and p["tiles"] == 32 * 32 and p["units"] == sms // 2
    assert p["waves"] == -(-1024 // (sms // 2))
    assert p["stream_k_tiles"] == 1024 - 13 * 76
    assert p["effective_waves"] == pytest.approx(13.5)
    assert p["pack_a"] == 0 and p["pack_b"] == 0
    # 4096^3: 256 tiles = 3 whole waves + 28; the 28 tail tiles split into k-halves on 56 pairs
    # (both halves add into C by TMA reduce-add, a few microseconds), 3.5 waves of time
    p = tct.gemm_f16_f32_plan(4096, 4096, 4096, num_sms=sms)
    assert (p["cta_group"], p["tile_n"], p["waves"], p["stream_k_tiles"]) == (2, 256, 4, 28)
    assert p["effective_waves"] == 3.5
    # 6144^3: 576 = 7 waves + 44 tiles on 76 pairs: 32 helpers take the second parts of 2
    # tail tiles each, so the owners keep ceil(2 * 96 / 3) = 64 of the 96 k-blocks
    p = tct.gemm_f16_f32_plan(6144, 6144, 6144, num_sms=sms)
    assert (p["waves"], p["stream_k_tiles"], p["split_kb"], p["split_parts_per_unit"]) == (8, 44, 64, 2)
    assert p["effective_waves"] == pytest.approx(7 + 64 / 96)
    p = tct.gemm_f16_f32_plan(4096, 4096, 16384, num_sms=sms)
    assert p["stream_k_tiles"] == 256 - 3 * 76 and p["effective_waves"] == 3.5
    p = tct.gemm_f16_f32_plan(4096, 4096, 16384, num_sms=sms, stream_k=1)
    assert p["stream_k_tiles"] == 0 and p["effective_waves"] == 4
    # the skinny, bandwidth-bound shape keeps at least 128 of the 152 SMs streaming B
    p = tct.gemm_f16_f32_plan(128, 16384, 16384, num_sms=sms)
    busy = p["cta_group"] * min(p["units"], p["tiles"] * (2 if p["stream_k_tiles"] else 1))
    assert busy >= 128
    # rows of C that end inside a 16-byte unit cannot be written by TMA: their split tiles
    # would combine through workspace (a helper takes one part, at a higher fixed cost), so
    # the same tile grid that splits with N % 4 == 0 keeps whole waves with N % 4 != 0
    p = tct.gemm_f16_f32_plan(6144, 6140, 6144, num_sms=sms)
    assert (p["stream_k_tiles"], p["split_parts_per_unit"]) == (44, 2)
    for n in (6142, 6143):
        p = tct.gemm_f16_f32_plan(6144, n, 6144, num_sms=sms)
        assert p["tiles"] == 576 and p["stream_k_tiles"] == 0
    assert tct.gemm_f16_f32_plan(4096, 4092, 4096, num_sms=sms)["stream_k_tiles"] == 28
    assert tct.gemm_f16_f32_plan(4096, 4094, 4096, num_sms=sms)["stream_k_tiles"] == 0
    # stream-K ranges where the k-loop is long against the tile count (measured 1.7x faster
    # than the two-part split at 256x256x65536); whole tiles for the under-filled single waves,
    # where each chain link costs about what it saves
    for shape in ((256, 256, 65536), (128, 512, 32768), (512, 512, 16384)):
        assert tct.gemm_f16_f32_plan(*shape, num_sms=sms)["split_form"] == 2, shape
    for shape in ((1792, 1792, 1792), (2048, 2048, 2048), (16384, 16384, 4096)):
        assert tct.gemm_f16_f32_plan(*shape, num_sms=sms)["split_form"] == 0, shape
    # wave quantisation decides the tile width: 1792^3 fills one wave better with 70 pair tiles
    # of 256x192 than with 49 of 256x256 (measured 19.5 against 20.5 us); 1793^3 (80 tiles of
    # 192 columns, more than the 76 pairs) and 2048^3 (64 tiles of 256) keep 256 columns
    assert (tct.gemm_f16_f32_plan(1792, 1792, 1792, num_sms=sms)["tile_n"],
            tct.gemm_f16_f32_plan(1792, 1792, 1792, num_sms=sms)["tiles"]) == (192, 70)
    for shape in ((1793, 1793, 1793), (2048, 2048, 2048), (4096, 4096, 4096), (8192, 8192, 8192)):
        assert tct.gemm_f16_f32_plan(*shape, num_sms=sms)["tile_n"] == 256, shape
    # the skinny, bandwidth-bound shape: among plans within 5% of the HBM time, the one whose
    # tiles move the fewest operand bytes from L2 (1-CTA 128x256 tiles, split in k-halves)
    p = tct.gemm_f16_f32_plan(128, 16384, 16384, num_sms=sms)
    assert (p["cta_group"], p["tile_n"], p["split_form"], p["stream_k_tiles"]) == (1, 256, 1, 64)
    for shape in ((4096, 4096, 4096), (8192, 8192, 8192), (1024, 1024, 8192)):
        assert tct.gemm_f16_f32_plan(*shape, num_sms=sms)["split_form"] == 1, shape
    # ragged leading dimensions are repacked before TMA
    p = tct.gemm_f16_f32_plan(17, 4097, 31, num_sms=sms)
    assert p["pack_a"] == 1 and p["pack_b"] == 1
    p = tct.gemm_f16_f32_plan(300, 200, 150, num_sms=sms)
    assert p["pack_a"] == 1 and p["pack_b"] == 0
    # explicit options are honoured
    p = tct.gemm_f16_f32_plan(4096, 4096, 4096, num_sms=sms, tile_n=256, stages=3, group_m=16, max_ctas=100)
    assert (p["tile_n"], p["stages"], p["group_m"], p["grid"]) == (256, 3, 16, 100)
    p = tct.gemm_f16_f32_plan(4096, 4096, 4096, num_sms=sms, cta_group=1, tile_n=256)
    assert (p["cta_group"], p["tile_m"], p["stages"], p["grid"]) == (1, 128, 4, 152)
    # every compiled variant's shared-memory ring fits the 227 KB limit
    for cg, tn, st in ((1, 256, 2), (1, 256, 3), (1, 256, 4), (1, 128, 4), (1, 128, 6), (2, 192, 6),
                       (2, 256, 3), (2, 256, 4), (2, 256, 5), (2, 256, 6), (2, 128, 6), (2, 128, 8)):
        p = tct.gemm_f16_f32_plan(4096, 4096, 4096, num_sms=sms, cta_group=cg, tile_n=tn, stages=st)
        assert (p["cta_group"], p["tile_n"], p["stages"]) == (cg, tn, st)
        assert 0 < p["smem_bytes"] <= 227 * 1024
    with pytest.raises(tct.GemmError):
        tct.gemm_f16_f32_plan(4096, 4096, 4096, num_sms=sms, cta_group=2, stages=2)


@pytest.mark.parametrize("shape,opts", [
    ((8192, 8192, 8192), {}), ((4096, 4096, 4096), {}), ((4096, 4096, 4096), {"stream_k": 1}),
    ((128, 16384, 16384), {}), ((1000, 1100, 700), {"stream_k": 2}), ((777, 1500, 515), {"stream_k": 2, "cta_group": 1}),
    ((300, 200, 150), {"stream_k": 2}), ((1, 1000, 640), {"stream_k": 2, "cta_group": 1, "tile_n": 128}),
    ((2000, 3000, 5000), {"stream_k": 2, "max_ctas": 50}), ((1792, 1792, 1792), {}), ((6144, 6144, 6144), {}),
    ((3072, 3072, 3072), {"stream_k": 2}), ((2048, 2048, 2048), {"stream_k": 2}), ((1792, 1792, 1792), {"stream_k": 2}),
    ((5000, 7000, 3000), {"stream_k": 2, "cta_group": 1, "tile_n": 128}),
])
def test_work_items_cover_every_k_block_once(tct_lib, shape, opts):
    """The library's own work split: each (tile, k-block) pair of the plan belongs to exactly
    one work item of one unit; every split tile has exactly one owner (its first split_kb
    k-blocks, mode 1) and one helper for the rest (mode 2), sharing one part slot; a helper
    takes split_parts_per_unit second parts at most, and no unit's k-blocks exceed the
    owner's share of the tail."""
    M, N, K = shape
    sms = 152
    p = tct.gemm_f16_f32_plan(M, N, K, num_sms=sms, **opts)
    kb = -(-K // 64)
    seen = {}
    owners, writers = {}, {}
    for u in range(p["units"]):
        idx = 0
        while True:
            it = tct.gemm_f16_f32_work_item(M, N, K, sms, u, idx, **opts)
            if it is None:
                break
            tile, kb0, kb1, mode, part = it["tile"], it["kb0"], it["kb1"], it["mode"], it["part"]
            assert 0 <= tile < p["tiles"] and 0 <= kb0 < kb1 <= kb
            if mode == tct.WORK_STORE:
                assert (kb0, kb1) == (0, kb) and part == -1
            else:
                assert tile >= p["tiles"] - p["stream_k_tiles"]
                book = owners if mode == tct.WORK_FIXUP else writers
                assert tile not in book
                book[tile] = (u, part, kb0, kb1)
            for k in range(kb0, kb1):
                assert (tile, k) not in seen
                seen[(tile, k)] = u
            idx += 1
    assert len(seen) == p["tiles"] * kb
    assert set(owners) == set(writers) and len(owners) == p["stream_k_tiles"]
    for tile, (u, part, kb0, kb1) in owners.items():
        wu, wpart, wkb0, wkb1 = writers[tile]
        assert wu != u and wpart == part and kb0 == 0 and kb1 == wkb0 and wkb1 == kb
    assert sorted(v[1] for v in owners.values()) == list(range(p["stream_k_tiles"]))
    if p["stream_k_tiles"]:
        per_helper = {}
        for tile, (wu, wpart, wkb0, wkb1) in writers.items():
            assert wkb0 == p["split_kb"]
            per_helper[wu] = per_helper.get(wu, 0) + (wkb1 - wkb0)
        assert max(per_helper.values()) <= p["split_parts_per_unit"] * (kb - p["split_kb"]) <= p["split_kb"]


STREAM_K_PLANS = [
    ((1792, 1792, 1792), {"stream_k": 3}), ((2048, 2048, 2048), {"stream_k": 3}),
    ((1792, 1796, 1793), {"stream_k": 3}), ((3072, 3072, 3072), {"stream_k": 3}),
    ((4096, 4096, 4096), {"stream_k": 3}), ((8192, 8192, 8192), {"stream_k": 3}),
    ((128, 16384, 16384), {"stream_k": 3}), ((128, 16384, 16384), {"stream_k": 3, "cta_group": 2}),
    ((256, 256, 4096), {"stream_k": 3}), ((300, 200, 150), {"stream_k": 3}),
    ((1, 1000, 64 * 40), {"stream_k": 3, "cta_group": 1, "tile_n": 128}),
    ((6144, 6144, 6144), {"stream_k": 3}), ((1000, 1100, 700), {"stream_k": 3, "max_ctas": 30}),
]


@pytest.mark.parametrize("shape,opts", STREAM_K_PLANS)
def test_stream_k_work_items(tct_lib, shape, opts):
    """Stream-K plans: each (tile, k-block) pair belongs to exactly one item of one unit; the
    whole waves come first; every unit's stream-K range is one contiguous, non-empty run of
    iterations in tile order, the ranges differ in length by at most one and together cover
    the stream-K tiles; only a unit's first piece starts inside a tile and only its last ends
    inside one; a tile's pieces lie on consecutive units, in k order, and number at most the
    plan's split_parts_per_unit."""
    M, N, K = shape
    sms = 152
    p = tct.gemm_f16_f32_plan(M, N, K, num_sms=sms, **opts)
    assert p["split_form"] == 2 and p["stream_k_tiles"] > 0 and 2 <= p["sk_units"] <= p["units"]
    kb = -(-K // 64)
    dp_tiles = p["tiles"] - p["stream_k_tiles"]
    assert dp_tiles % p["units"] == 0
    seen = {}
    pieces = {}
    lengths = []
    for u in range(p["units"]):
        idx = 0
        sk_items = []
        while True:
            it = tct.gemm_f16_f32_work_item(M, N, K, sms, u, idx, **opts)
            if it is None:
                break
            tile, kb0, kb1, mode = it["tile"], it["kb0"], it["kb1"], it["mode"]
            assert 0 <= kb0 < kb1 <= kb
            if idx < dp_tiles // p["units"]:
                assert mode == tct.WORK_STORE and tile == u + idx * p["units"] and (kb0, kb1) == (0, kb)
            else:
                assert tile >= dp_tiles
                sk_items.append((tile, kb0, kb1, mode, it["part"]))
            for k in range(kb0, kb1):
                assert (tile, k) not in seen
                seen[(tile, k)] = u
            idx += 1
        if u >= p["sk_units"]:
            assert not sk_items
            continue
        assert sk_items, f"unit {u} has an empty stream-K range"
        flat = [(t - dp_tiles) * kb + k for (t, k0, k1, _, _) in sk_items for k in range(k0, k1)]
        assert flat == list(range(flat[0], flat[0] + len(flat)))  # contiguous, in order
        lengths.append((flat[0], len(flat)))
        for j, (t, k0, k1, mode, part) in enumerate(sk_items):
            whole = (k0, k1) == (0, kb)
            assert mode == (tct.WORK_STORE if whole else tct.WORK_CHAIN)
            assert part == (-1 if whole else u)
            if k0 > 0:
                assert j == 0
            if k1 < kb:
                assert j == len(sk_items) - 1
            if not whole:
                pieces.setdefault(t, []).append((u, k0, k1))
    assert len(seen) == p["tiles"] * kb
    starts = [a for a, _ in lengths]
    assert starts == sorted(starts) and starts[0] == 0
    assert max(n for _, n in lengths) - min(n for _, n in lengths) <= 1
    assert sum(n for _, n in lengths) == p["stream_k_tiles"] * kb
    assert min(n for _, n in lengths) == p["split_kb"]
    for t, ps in pieces.items():
        units = [u for u, _, _ in ps]
        assert units == list(range(units[0], units[0] + len(units)))
        assert ps[0][1] == 0 and ps[-1][2] == kb
        assert all(ps[i][2] == ps[i + 1][1] for i in range(len(ps) - 1))
        assert len(ps) <= p["split_parts_per_unit"]


def test_stream_k_needs_the_reduce_add_path(tct_lib):
    """Stream-K combines pieces by TMA reduce-add into C: it is only planned for the plain
    FP32 epilogue on a C whose rows are whole 16-byte units; asked for otherwise, the plan
    is rejected."""
    sms = 152
    assert tct.gemm_f16_f32_plan(2048, 2048, 2048, num_sms=sms, stream_k=3)["split_form"] == 2
    with pytest.raises(tct.GemmError):
        tct.gemm_f16_f32_plan(2048, 2046, 2048, num_sms=sms, stream_k=3)


def test_stream_k_plans_cover_both_combinations(tct_lib):
    """The stream-K plans above include tiles of at most two pieces (added into C in either
    order) and longer chains (added in a fixed order), so both combinations are exercised."""
    pieces = {tct.gemm_f16_f32_plan(*shape, num_sms=152, **opts)["split_parts_per_unit"] for shape, opts in STREAM_K_PLANS}
    assert min(pieces) <= 2 < max(pieces)

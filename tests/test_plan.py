"""The planner (a pure host function of the C library) and the kernel's index
arithmetic, checked on the CPU for every workload shape and for forced
configurations, before anything runs on a GPU."""
from __future__ import annotations

import itertools

import pytest

import kernel_model

SM = 152  # GB300; the planner takes the SM count as an argument
WORKLOADS = [
    (256, 512), (7168, 16384), (18432, 7168), (4096, 4096), (14336, 4096), (4096, 14336),
    (28672, 8192), *itertools.product([1024, 4099, 18433, 65536], [1000, 4096, 7169, 16384]),
    (57344, 7168), (1, 1), (1, 7), (3, 9), (1, 100000), (2, 2 ** 20), (100000, 8),
]
MAX_SMEM = 232448


@pytest.mark.parametrize("n,k", WORKLOADS)
@pytest.mark.parametrize("dtype", [0, 1, 2, 3])
@pytest.mark.parametrize("aligned", [True, False])
@pytest.mark.parametrize("sm", [SM, 148])
def test_plan_invariants(gemv_lib, n, k, dtype, aligned, sm):
    cfg = gemv_lib.gemv_plan(n, k, dtype, aligned, sm)
    W, R, Sw, Sg = cfg["warps_per_cta"], cfg["rows_per_warp"], cfg["warp_split"], cfg["grid_split"]
    assert W in (4, 8, 16) and R in (1, 2, 4) and W % Sw == 0
    assert cfg["variant"] in (3, 4)
    kseg = cfg["k_segment"]
    assert Sg * kseg >= k and (Sg - 1) * kseg < k
    if Sg > 1:
        assert kseg % 8 == 0
    assert cfg["ctas"] == cfg["row_blocks"] * Sg >= 1
    assert cfg["smem_bytes"] <= MAX_SMEM
    assert cfg["launches"] == (2 if Sg > 1 else 1)
    # persistent grid: never more CTAs than can be resident at once
    cps = min(32 // W, 233472 // (cfg["smem_bytes"] + 1024))
    assert cfg["ctas"] <= max(sm * cps, Sg * 8)


def test_plan_shapes_of_interest(gemv_lib):
    """The plans measured fastest (or within 3 %) on GB300 for the workload
    shapes, back to back with programmatic dependent launch."""
    big = gemv_lib.gemv_plan(7168, 16384, 0, True, SM)
    assert big["grid_split"] == 1 and big["warp_split"] == 4 and big["variant"] == 3
    assert big["warps_per_cta"] == 16 and big["rows_per_warp"] == 2 and big["unroll"] == 4
    # rows split over warps take two rows per warp and twice the split
    p = gemv_lib.gemv_plan(4096, 14336, 1, True, SM)
    assert (p["warp_split"], p["rows_per_warp"], p["unroll"]) == (4, 2, 4)
    p = gemv_lib.gemv_plan(256, 262144, 0, True, SM)
    assert (p["grid_split"], p["warp_split"], p["rows_per_warp"], p["unroll"]) == (8, 8, 2, 4)
    p = gemv_lib.gemv_plan(18432, 7168, 1, True, SM)
    assert (p["warp_split"], p["rows_per_warp"], p["unroll"]) == (1, 2, 4)
    p = gemv_lib.gemv_plan(14336, 4096, 1, True, SM)
    assert (p["warp_split"], p["rows_per_warp"], p["unroll"]) == (1, 1, 8)
    p = gemv_lib.gemv_plan(4096, 4096, 1, True, SM)
    assert (p["warp_split"], p["rows_per_warp"], p["ctas"]) == (1, 1, 304)  # every slot: part-filled tiles
    assert gemv_lib.gemv_plan(4099, 1000, 0, True, SM)["ctas"] == 257        # short rows: whole tiles only
    assert gemv_lib.gemv_plan(1024, 1000, 0, True, SM)["ctas"] == 64
    assert gemv_lib.gemv_plan(4099, 7169, 1, False, SM)["ctas"] == 304
    p = gemv_lib.gemv_plan(1024, 4096, 0, True, SM)
    assert (p["warp_split"], p["unroll"]) == (4, 4)
    p = gemv_lib.gemv_plan(256, 512, 0, True, SM)
    assert (p["warps_per_cta"], p["warp_split"], p["rows_per_warp"], p["unroll"], p["ctas"]) == (16, 1, 1, 4, 16)
    assert gemv_lib.gemv_plan(65536, 4096, 1, True, SM)["warp_split"] == 1
    tiny_n = gemv_lib.gemv_plan(16, 16384, 0, True, SM)
    assert tiny_n["warp_split"] * tiny_n["grid_split"] > 1  # rows are split to fill the GPU
    huge_k = gemv_lib.gemv_plan(2, 2 ** 20, 1, True, SM)
    assert huge_k["grid_split"] >= 32 and huge_k["k_segment"] <= 32768


@pytest.mark.parametrize("cfg", [
    {"variant": 1, "rows_per_warp": 4}, {"variant": 1, "warps_per_cta": 4, "warp_split": 4},
    {"variant": 1, "grid_split": 3}, {"variant": 1, "warps_per_cta": 8, "warp_split": 2, "grid_split": 2},
    {"variant": 1, "ctas": 7}, {"variant": 1, "ctas": 1}, {"variant": 1, "warps_per_cta": 16, "warp_split": 16},
    {"warps_per_cta": 4, "warp_split": 4}, {"grid_split": 3}, {"warps_per_cta": 8, "warp_split": 2, "grid_split": 2},
    {"ctas": 16}, {"warps_per_cta": 16, "warp_split": 16}, {"rows_per_warp": 2, "unroll": 4},
])
def test_forced_configs_are_honoured(gemv_lib, cfg):
    """(1000 x 4096: see also the shapes of the GPU forced-config test below.)"""
    out = gemv_lib.gemv_plan(1000, 4096, 0, True, SM, config=cfg)
    for key, v in cfg.items():
        if key == "ctas":
            assert out["ctas"] == (v // out["grid_split"]) * out["grid_split"]
        else:
            assert out[key] == v


@pytest.mark.parametrize("cfg", [
    {"variant": 5}, {"rows_per_warp": 3}, {"warps_per_cta": 12}, {"warps_per_cta": 8, "warp_split": 3},
    {"grid_split": 65537}, {"variant": 2, "rows_per_warp": 2}, {"rows_per_warp": 2, "unroll": 8},
])
def test_invalid_forced_configs_rejected(gemv_lib, cfg):
    with pytest.raises(gemv_lib.GemvError) as ei:
        gemv_lib.gemv_plan(1000, 4096, 0, True, SM, config=cfg)
    assert ei.value.status == gemv_lib.GEMV_ERR_CONFIG


def test_aligned_variant_refused_for_ragged_k(gemv_lib):
    with pytest.raises(gemv_lib.GemvError):
        gemv_lib.gemv_plan(100, 4097, 0, True, SM, config={"variant": 1})
    with pytest.raises(gemv_lib.GemvError):
        gemv_lib.gemv_plan(100, 4096, 0, False, SM, config={"variant": 1})


# ------------------------------------------------ index-arithmetic replay --

SMALL = [(1, 1), (1, 8), (2, 7), (3, 9), (5, 17), (13, 31), (17, 64), (33, 100), (64, 512), (7, 1000),
         (40, 257), (129, 33), (3, 4099)]


@pytest.mark.parametrize("n,k", SMALL)
@pytest.mark.parametrize("base_off", [0, 1, 3, 7])
@pytest.mark.parametrize("forced", [None, {"warps_per_cta": 4, "warp_split": 2},
                                    {"grid_split": 3}, {"warps_per_cta": 8, "warp_split": 4, "grid_split": 2},
                                    {"ctas": 3}, {"warps_per_cta": 16, "warp_split": 16}])
def test_general_variant_index_replay(gemv_lib, n, k, base_off, forced):
    try:
        cfg = gemv_lib.gemv_plan(n, k, 0, False, SM, config={**(forced or {}), "variant": 2})
    except gemv_lib.GemvError:
        pytest.skip("configuration not valid for this shape")
    assert cfg["variant"] == 2
    kernel_model.replay(n, k, cfg, base_off=base_off)


@pytest.mark.parametrize("n,k", [(1, 8), (3, 16), (5, 64), (17, 256), (64, 512), (33, 1000), (7, 4096),
                                 (129, 40), (300, 24)])
@pytest.mark.parametrize("forced", [None, {"rows_per_warp": 2}, {"rows_per_warp": 4},
                                    {"rows_per_warp": 4, "warps_per_cta": 4, "warp_split": 2},
                                    {"grid_split": 3}, {"ctas": 2, "rows_per_warp": 2},
                                    {"warps_per_cta": 16, "warp_split": 8, "grid_split": 2}])
def test_aligned_variant_index_replay(gemv_lib, n, k, forced):
    try:
        cfg = gemv_lib.gemv_plan(n, k, 1, True, SM, config={**(forced or {}), "variant": 1})
    except gemv_lib.GemvError:
        pytest.skip("configuration not valid for this shape")
    assert cfg["variant"] == 1
    kernel_model.replay(n, k, cfg, base_off=0)


@pytest.mark.parametrize("n,k,aligned", [(256, 512, True), (1024, 1000, True), (4099, 1000, True),
                                         (1024, 7169, False), (300, 7169, False)])
def test_planner_choice_replay_medium(gemv_lib, n, k, aligned):
    cfg = gemv_lib.gemv_plan(n, k, 0, aligned, SM)
    kernel_model.replay(n, k, cfg, base_off=0 if aligned else 3)


# ------------------------------------------------------------ tiles variant --

TILES_FORCED = [None, {"warp_split": 2}, {"warp_split": 4, "warps_per_cta": 8},
                {"rows_per_warp": 2, "unroll": 4}, {"rows_per_warp": 4, "unroll": 2},
                {"rows_per_warp": 1, "unroll": 4}, {"grid_split": 3}, {"ctas": 8},
                {"warps_per_cta": 16, "warp_split": 16}, {"warps_per_cta": 4, "warp_split": 2, "grid_split": 2}]


@pytest.mark.parametrize("n,k", SMALL + [(64, 512), (33, 1000), (300, 24), (2, 4096), (1, 2049)])
@pytest.mark.parametrize("base_off", [0, 1, 6])
@pytest.mark.parametrize("forced", TILES_FORCED)
def test_tiles_index_replay(gemv_lib, n, k, base_off, forced):
    cfg_in = dict(forced or {})
    cfg_in["variant"] = 3
    aligned = base_off == 0
    try:
        cfg = gemv_lib.gemv_plan(n, k, 0, aligned, SM, config=cfg_in)
    except gemv_lib.GemvError:
        pytest.skip("configuration not valid for this shape")
    kernel_model.replay(n, k, cfg, base_off=base_off)


@pytest.mark.parametrize("n,k", WORKLOADS)
@pytest.mark.parametrize("aligned", [True, False])
def test_tiles_plan_invariants(gemv_lib, n, k, aligned):
    cfg = gemv_lib.gemv_plan(n, k, 1, aligned, SM, config={"variant": 3})
    W, S, C, Sg = cfg["warps_per_cta"], cfg["warp_split"], cfg["row_blocks"], cfg["grid_split"]
    ncls = 1 if aligned and k % 8 == 0 else 8
    assert W % S == 0 and C % ncls == 0 and C >= ncls and cfg["ctas"] == C * Sg
    assert Sg * cfg["k_segment"] >= k and (Sg - 1) * cfg["k_segment"] < k
    assert cfg["smem_bytes"] <= MAX_SMEM
    nt = -(-cfg["k_segment"] // 8) + (0 if ncls == 1 else 1)
    # row slices of at most 1024 blocks (16 KB) plus the <= 32 blocks the
    # kernel folds into a slice's last step, unless the row is too long for 16 warps
    assert -(-nt // S) <= 1024 + 32 or S == W
    # slices are not cut below 128 blocks to fill the GPU
    assert S == 1 or -(-nt // S) >= 128 or -(-nt // (S // 2)) > 1024 + 32


@pytest.mark.parametrize("n,k,aligned", [(256, 512, True), (1024, 1000, True), (130, 7169, False),
                                         (77, 4099, False), (1000, 600, False)])
def test_tiles_planner_choice_replay_medium(gemv_lib, n, k, aligned):
    cfg = gemv_lib.gemv_plan(n, k, 0, aligned, SM, config={"variant": 3})
    kernel_model.replay(n, k, cfg, base_off=0 if aligned else 5)


@pytest.mark.parametrize("off", range(8))
@pytest.mark.parametrize("j0,seglen,k", [(0, 37, 37), (8, 20, 40), (16, 7169 - 16, 7169), (0, 8, 8)])
def test_shifted_staging_model(off, j0, seglen, k):
    """The vector-plus-shift staging equals the definition
    as[x] = a[j0 + x - off] for off <= x < off + seglen, 0 elsewhere."""
    import numpy as np
    a = np.arange(1, k + 1, dtype=np.int64)
    as_elems = -(-(seglen + 24) // 8) * 8
    got = kernel_model.staged_shifted(a, j0, seglen, off, as_elems)
    want = np.zeros(as_elems, dtype=np.int64)
    for x in range(as_elems):
        if off <= x < off + seglen:
            want[x] = a[j0 + x - off]
    assert (got == want).all()


@pytest.mark.parametrize("shifted", [False, True])
@pytest.mark.parametrize("block", [32, 256, 512, 1024])
@pytest.mark.parametrize("nvec", [0, 1, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1023, 1024, 1025, 1056, 2048, 2049,
                                  2051, 4096, 4100])
def test_staging_schedule(nvec, block, shifted):
    """Every staged vector written exactly once by the paired-then-single
    staging loop, and the pairs taken wherever a thread has two vectors."""
    most = kernel_model.staging_schedule(nvec, block, shifted)
    assert most == (0 if shifted or nvec <= block else -(-(nvec - block) // (2 * block)))


@pytest.mark.parametrize("n,k,ldb", [(5, 17, 24), (9, 64, 72), (9, 64, 67), (33, 100, 100), (17, 7, 8), (3, 4099, 5000),
                                     (40, 256, 264), (7, 1000, 1003)])
@pytest.mark.parametrize("base_off", [0, 3])
@pytest.mark.parametrize("forced", [None, {"warp_split": 2}, {"grid_split": 3}, {"rows_per_warp": 2, "unroll": 4}])
def test_tiles_index_replay_strided(gemv_lib, n, k, ldb, base_off, forced):
    """Row-strided B (ldb >= k): rows start at i * ldb; aligned only when the
    base, k and ldb all allow it."""
    cfg_in = dict(forced or {})
    cfg_in["variant"] = 3
    aligned = base_off == 0 and ldb % 8 == 0
    try:
        cfg = gemv_lib.gemv_plan(n, k, 0, aligned, SM, config=cfg_in)
    except gemv_lib.GemvError:
        pytest.skip("configuration not valid for this shape")
    kernel_model.replay(n, k, cfg, base_off=base_off, ldb=ldb)


@pytest.mark.parametrize("bh,dk,dv,es", [(3, 128, 128, 2), (2, 64, 64, 4), (5, 17, 8, 2), (1, 1, 2048, 2),
                                         (2, 100, 1024, 4), (4, 256, 24, 2), (1, 0, 64, 2), (7, 64, 64, 2),
                                         (37, 16, 64, 2), (11, 5, 24, 2), (6, 3, 40, 4)])
@pytest.mark.parametrize("grid", [1, 3, None])
def test_gla_index_replay(bh, dk, dv, es, grid):
    kernel_model.replay_gla(bh, dk, dv, es, grid=grid)


def test_gla_balanced_grid():
    """The GLA grid: never above the resident cap, every CTA gets a round,
    no CTA runs more rounds than the cap forces (ceil(units / cap)), the
    round counts differ by at most one, and it stays at the cap when
    balancing would drop more than a fifth of it."""
    bg = kernel_model.gla_balanced_grid
    assert bg(2048, 608) == 512 and bg(4096, 608) == 586 and bg(2048, 456) == 410 and bg(100, 608) == 100
    assert bg(1024, 456) == 456 and bg(1024, 608) == 512
    for units in list(range(1, 400)) + [2047, 2048, 2049, 4096, 65536, 10**6 + 7]:
        for cap in (1, 3, 152, 304, 456, 608, 1216):
            grid = bg(units, cap)
            assert 1 <= grid <= min(units, cap)
            assert grid == min(units, cap) or 5 * grid >= 4 * cap
            per = [len(range(b, units, grid)) for b in range(grid)] if units < 5000 else None
            if per is not None:
                assert min(per) >= 1 and max(per) == -(-units // cap) and max(per) - min(per) <= 1


@pytest.mark.parametrize("bh,dk,dv,es,cap", [(2048, 8, 64, 2, 608), (1031, 3, 16, 4, 152), (300, 16, 64, 2, 456)])
def test_gla_index_replay_balanced_grid(bh, dk, dv, es, cap):
    """The replay at the grid the host computes from a resident cap."""
    cpr = dv * es // 16
    G = kernel_model.gla_heads_per_cta(bh, dk, cpr)
    kernel_model.replay_gla(bh, dk, dv, es, grid=kernel_model.gla_balanced_grid(-(-bh // G), cap))
    kernel_model.replay_gla_warp(bh, dk, dv, es, grid=-(-kernel_model.gla_balanced_grid(bh, cap * 8) // 8))


@pytest.mark.parametrize("bh,dk,dv,es", [(3, 128, 128, 2), (2, 64, 64, 4), (5, 16, 8, 2), (9, 8, 256, 2),
                                         (2, 64, 128, 4), (4, 16, 24, 2), (7, 64, 64, 2), (37, 16, 64, 2),
                                         (11, 8, 24, 2), (6, 4, 40, 4), (300, 16, 64, 2), (1, 200, 64, 2)])
@pytest.mark.parametrize("grid", [1, 3, None])
def test_gla_pipe_index_replay(bh, dk, dv, es, grid):
    kernel_model.replay_gla_pipe(bh, dk, dv, es, grid=grid)


def test_gla_pipe_choice():
    """The pipelined layout applies to rows of whole 16-byte chunks and
    heads within 32 KiB; the workload shapes 2048 x 128 x 128 bf16, 4096 x
    64 x 64 fp16 and 16384 x 16 x 64 fp16 take it with 1, 4 and 16 heads
    per round, in buffers of which 2 CTAs fit an SM (228 KB, 1 KB reserved
    per CTA)."""
    ok, hp = kernel_model.gla_pipe_ok, kernel_model.gla_pipe_heads_per_cta
    assert ok(128, 128, 2) and ok(64, 64, 2) and ok(16, 64, 2) and ok(64, 64, 4)
    assert not ok(128, 128, 4) and not ok(256, 256, 2) and not ok(5, 64, 2) and not ok(0, 64, 2)
    assert hp(2048, 128, 128, 2) == 1 and hp(4096, 64, 64, 2) == 4 and hp(16384, 16, 64, 2) == 16
    assert hp(8192, 64, 64, 4) == 2
    auto = kernel_model.gla_auto_is_pipe
    assert auto(128, 128, 2) and auto(64, 64, 2) and auto(16, 64, 2) and not auto(128, 128, 4)
    assert not auto(256, 256, 2) and not auto(5, 64, 2)
    for bh, dk, dv, es in [(2048, 128, 128, 2), (4096, 64, 64, 2), (16384, 16, 64, 2), (2048, 64, 64, 4),
                           (5, 8, 2048, 2), (64, 2048, 8, 2)]:
        if ok(dk, dv, es):
            smem = kernel_model.gla_pipe_smem(hp(bh, dk, dv, es), dk, dv, es)
            assert 2 * (smem + 1024) <= 233472, (bh, dk, dv, smem)


@pytest.mark.parametrize("cpr,vec", [(16, 8), (8, 8), (32, 8), (4, 8), (2, 8), (1, 8), (3, 8), (5, 8), (16, 4),
                                     (32, 4), (8, 4), (2, 4)])
def test_gla_partial_stores_conflict_free(cpr, vec):
    """The 16-byte partial stores, in the order ``store_partials`` issues
    them, hit 8 distinct bank groups in every 8-lane phase (the naive order
    for 8 floats per lane conflicts 2-way)."""
    dv = cpr * vec
    assert kernel_model.gla_partial_store_conflicts(cpr, vec, dv) == 0


def test_gla_heads_per_cta_choice():
    """Small heads are processed several per CTA round (about 4 rows per
    thread), large ones one per round."""
    hp = kernel_model.gla_heads_per_cta
    assert kernel_model.gla_rows_in_flight(64, 8) == 8 and kernel_model.gla_rows_in_flight(128, 16) == 4
    assert hp(4096, 64, 8) == 4 and hp(16384, 16, 8) == 16 and hp(2048, 128, 16) == 1
    assert hp(1024, 256, 32) == 1 and hp(1, 16, 8) == 1 and hp(3, 16, 8) == 2
    assert hp(4096, 64, 8, rows_in_flight=4) == 2


# ------------------------------------------------------------- bulk variant --

BULK_FORCED = [{}, {"stages": 2}, {"stages": 3, "unroll": 4}, {"unroll": 8, "stages": 2}, {"warp_split": 2},
               {"warps_per_cta": 8, "warp_split": 4, "stages": 3}, {"grid_split": 3}, {"ctas": 8},
               {"warps_per_cta": 4, "warp_split": 2, "grid_split": 2, "stages": 5}, {"stages": 8, "unroll": 4}]


@pytest.mark.parametrize("n,k", [(1, 1), (3, 9), (17, 7), (64, 512), (33, 1000), (9, 5000), (40, 4099),
                                 (5, 16384), (2, 33000), (300, 24), (130, 2056)])
@pytest.mark.parametrize("base_off", [0, 1, 6])
@pytest.mark.parametrize("forced", BULK_FORCED)
def test_bulk_index_replay(gemv_lib, n, k, base_off, forced):
    """Ring replay of the bulk kernel: several chunks per row slice, rings that
    wrap, unaligned rows, split-K."""
    cfg_in = dict(forced)
    cfg_in["variant"] = 4
    aligned = base_off == 0
    try:
        cfg = gemv_lib.gemv_plan(n, k, 0, aligned, SM, config=cfg_in)
    except gemv_lib.GemvError:
        pytest.skip("configuration not valid for this shape")
    assert cfg["variant"] == 4 and cfg["rows_per_warp"] == 1
    for key in ("stages", "unroll", "warp_split", "warps_per_cta"):
        if key in forced:
            assert cfg[key] == forced[key]
    kernel_model.replay(n, k, cfg, base_off=base_off)


@pytest.mark.parametrize("n,k,ldb", [(5, 17, 24), (9, 64, 67), (17, 7, 8), (3, 4099, 5000), (7, 1000, 1003),
                                     (6, 3000, 3008)])
@pytest.mark.parametrize("base_off", [0, 3])
@pytest.mark.parametrize("forced", [{}, {"warp_split": 2, "stages": 2}, {"grid_split": 3}])
def test_bulk_index_replay_strided(gemv_lib, n, k, ldb, base_off, forced):
    cfg_in = dict(forced)
    cfg_in["variant"] = 4
    aligned = base_off == 0 and ldb % 8 == 0
    try:
        cfg = gemv_lib.gemv_plan(n, k, 0, aligned, SM, config=cfg_in)
    except gemv_lib.GemvError:
        pytest.skip("configuration not valid for this shape")
    kernel_model.replay(n, k, cfg, base_off=base_off, ldb=ldb)


@pytest.mark.parametrize("n,k", WORKLOADS)
@pytest.mark.parametrize("aligned", [True, False])
def test_bulk_plan_invariants(gemv_lib, n, k, aligned):
    cfg = gemv_lib.gemv_plan(n, k, 1, aligned, SM, config={"variant": 4})
    W, S, C, Sg, U, NS = (cfg[x] for x in ("warps_per_cta", "warp_split", "row_blocks", "grid_split", "unroll",
                                            "stages"))
    ncls = 1 if aligned and k % 8 == 0 else 8
    assert cfg["variant"] == 4 and cfg["rows_per_warp"] == 1 and U in (4, 8) and NS == 2
    assert W % S == 0 and C % ncls == 0 and C >= ncls and cfg["ctas"] == C * Sg
    assert Sg * cfg["k_segment"] >= k and (Sg - 1) * cfg["k_segment"] < k
    as_elems = -(-(cfg["k_segment"] + 24) // 8) * 8
    ring_off = -(-(as_elems * 2 + 8 * W) // 128) * 128
    assert cfg["smem_bytes"] == ring_off + W * NS * (512 * U + 8) <= MAX_SMEM
    assert cfg["l2_prefetch"] == 0
    # never more CTAs than are resident at once
    cps = min(32 // W, 233472 // (cfg["smem_bytes"] + 1024))
    assert cfg["ctas"] <= max(SM * cps, Sg * ncls)


@pytest.mark.parametrize("cfg", [{"variant": 4, "rows_per_warp": 2}, {"variant": 4, "unroll": 2},
                                 {"variant": 4, "stages": 1}, {"variant": 4, "stages": 9},
                                 {"variant": 4, "l2_prefetch": 1}, {"variant": 3, "stages": 2},
                                 {"variant": 1, "stages": 2}, {"stages": 3}])
def test_bulk_invalid_configs_rejected(gemv_lib, cfg):
    with pytest.raises(gemv_lib.GemvError) as ei:
        gemv_lib.gemv_plan(4096, 4096, 0, True, SM, config=cfg)
    assert ei.value.status == gemv_lib.GEMV_ERR_CONFIG


@pytest.mark.parametrize("aligned", [True, False])
def test_bulk_auto_choice(gemv_lib, aligned):
    """Unforced plans use the bulk variant (with its own plan) exactly for B
    of at least 768 MiB whose tiles plan has one warp per row and whose rows
    hold 6144 to 8191 elements; everything else is the tiles plan."""
    shapes = WORKLOADS + [(65536, 7169), (16384, 7169), (18432, 7168), (65536, 16384), (131072, 4096),
                          (98304, 7168), (262144, 2048), (57344, 8192), (65536, 8192), (131072, 6144),
                          (131072, 6143), (98304, 8191), (98304, 8192), (49152, 8000)]
    for n, k in shapes:
        auto = gemv_lib.gemv_plan(n, k, 0, aligned, SM)
        tiles = gemv_lib.gemv_plan(n, k, 0, aligned, SM, config={"variant": 3})
        if n * k * 2 >= (768 << 20) and tiles["warp_split"] <= tiles["rows_per_warp"] and 6144 <= k < 8192:
            assert auto["variant"] == 4, (n, k, aligned)
            assert auto == gemv_lib.gemv_plan(n, k, 0, aligned, SM, config={"variant": 4})
        else:
            assert auto == tiles and auto["variant"] == 3, (n, k, aligned)
    assert gemv_lib.gemv_plan(57344, 7168, 1, True, SM)["variant"] == 4
    assert gemv_lib.gemv_plan(65536, 7169, 0, False, SM)["variant"] == 4
    assert gemv_lib.gemv_plan(131072, 4096, 0, True, SM)["variant"] == 3
    assert gemv_lib.gemv_plan(57344, 8192, 0, True, SM)["variant"] == 3
    assert gemv_lib.gemv_plan(16384, 7169, 0, False, SM)["variant"] == 3
    assert gemv_lib.gemv_plan(7168, 16384, 0, True, SM)["variant"] == 3
    assert gemv_lib.gemv_plan(18432, 7168, 1, True, SM)["variant"] == 3


@pytest.mark.parametrize("n,k,base_off", [(16384, 7169, 0)])
def test_bulk_auto_plans_replay(gemv_lib, n, k, base_off):
    """A bulk plan of a workload shape, replayed in full (every CTA, warp
    and ring chunk)."""
    cfg = gemv_lib.gemv_plan(n, k, 0, base_off == 0, SM, config={"variant": 4})
    assert cfg["variant"] == 4
    kernel_model.replay(n, k, cfg, base_off=base_off)


@pytest.mark.parametrize("bh,dk,dv,es", [(3, 128, 128, 2), (2, 64, 64, 4), (5, 17, 8, 2), (9, 1, 256, 2),
                                         (2, 100, 128, 4), (4, 256, 24, 2), (1, 0, 64, 2), (33, 64, 64, 2),
                                         (17, 5, 48, 4)])
@pytest.mark.parametrize("grid", [1, 2, None])
def test_gla_warp_index_replay(bh, dk, dv, es, grid):
    kernel_model.replay_gla_warp(bh, dk, dv, es, grid=grid)


@pytest.mark.parametrize("n,k,base_off,R", [(18433, 1003, 3, 2), (19456, 512, 0, 2), (10007, 1003, 3, 1),
                                             (300, 100003, 5, 1), (12000, 2056, 0, 1)])
def test_default_plan_replay_two_rows_and_split_k(gemv_lib, n, k, base_off, R):
    """Default plans of the regimes the planner tuning introduced -- two rows
    per warp for many rows (aligned and unaligned; one row where two would
    leave more of the last round idle), split-K with 16 warps per row for
    few unaligned rows -- replayed in full."""
    cfg = gemv_lib.gemv_plan(n, k, 0, base_off == 0, SM)
    assert cfg["rows_per_warp"] == R
    kernel_model.replay(n, k, cfg, base_off=base_off)


@pytest.mark.parametrize("n,k,aligned", [(2, 3_000_000, True), (3, 5_000_001, False), (1, 2**31 - 1, False),
                                         (64, 2**22, True), (1, 2**31 - 8, True)])
def test_long_rows_plan(gemv_lib, n, k, aligned):
    """k up to INT32_MAX: as many 32768-column segments as k needs (up to
    65536), for both kernels."""
    for variant in (0, 4):
        cfg = gemv_lib.gemv_plan(n, k, 0, aligned, SM, config={"variant": variant} if variant else None)
        assert cfg["k_segment"] <= 32768 and cfg["grid_split"] * cfg["k_segment"] >= k
        assert (cfg["grid_split"] - 1) * cfg["k_segment"] < k
        assert cfg["launches"] == 2 and cfg["ctas"] == cfg["row_blocks"] * cfg["grid_split"]


@pytest.mark.parametrize("n,k,base_off", [(2, 3_000_000, 0), (3, 5_000_001, 3)])
def test_long_rows_replay(gemv_lib, n, k, base_off):
    for variant in (None, 4):
        cfg = gemv_lib.gemv_plan(n, k, 0, base_off == 0, SM, config={"variant": variant} if variant else None)
        kernel_model.replay(n, k, cfg, base_off=base_off)


@pytest.mark.parametrize("cfg", [{"variant": 3, "warp_split": 1, "rows_per_warp": 1, "unroll": 8},
                                 {"variant": 3, "warp_split": 1, "rows_per_warp": 2, "unroll": 4},
                                 {"variant": 3, "warp_split": 2, "rows_per_warp": 1, "unroll": 8}])
@pytest.mark.parametrize("base_off", [0, 3])
def test_folded_step_plans_replay(gemv_lib, cfg, base_off):
    """The forced plans of the folded-last-step GPU test, replayed in full
    before they run (row lengths of 32*U*m + {1, 2, 32, 33} blocks)."""
    for k in [1032, 1288, 2049, 2056, 2304, 2328, 4104, 4112, 4113]:
        p = gemv_lib.gemv_plan(300, k, 0, base_off == 0, SM, config=cfg)
        kernel_model.replay(300, k, p, base_off=base_off)


# The forced configurations of the GPU parity test, on its shape and on long
# rows, where the planner's own choices (two rows per warp with twice the
# split) would otherwise apply: every forced field but ctas and grid_split
# is kept as given.
GPU_FORCED = [
    {"variant": 2}, {"rows_per_warp": 2}, {"rows_per_warp": 4}, {"warps_per_cta": 4},
    {"warps_per_cta": 8, "warp_split": 8}, {"warps_per_cta": 16, "warp_split": 4}, {"grid_split": 2},
    {"grid_split": 5, "warp_split": 2}, {"ctas": 37, "rows_per_warp": 2}, {"variant": 3},
    {"variant": 3, "warp_split": 8}, {"variant": 3, "warp_split": 2, "warps_per_cta": 4},
    {"variant": 3, "warp_split": 2}, {"variant": 3, "warp_split": 1},
    {"variant": 3, "rows_per_warp": 2, "unroll": 4}, {"variant": 3, "grid_split": 4},
    {"variant": 3, "l2_prefetch": 1}, {"variant": 3, "l2_prefetch": 3, "warp_split": 2},
]


@pytest.mark.parametrize("cfg", GPU_FORCED)
@pytest.mark.parametrize("n,k", [(1537, 4096), (7168, 16384), (4096, 14336), (256, 262144)])
def test_forced_fields_kept(gemv_lib, cfg, n, k):
    try:
        out = gemv_lib.gemv_plan(n, k, 0, True, SM, config=cfg)
    except gemv_lib.GemvError as e:
        assert e.status == gemv_lib.GEMV_ERR_CONFIG
        return
    for key, v in cfg.items():
        if key not in ("ctas", "grid_split"):
            assert out[key] == v, (key, out)


@pytest.mark.parametrize("variant", [None, 3, 4])
def test_ragged_tail_plans_replay(gemv_lib, variant):
    """The plans of the GPU ragged-tail test (every n and k in 1..17,
    31..33, 255..257, 4099, 7169), replayed in full where small."""
    sizes = list(range(1, 18)) + [31, 32, 33, 255, 256, 257, 4099, 7169]
    cfg = {"variant": variant} if variant else None
    for n, k in itertools.product(sizes, sizes):
        if n > 257 and k > 257:
            continue
        p = gemv_lib.gemv_plan(n, k, 0, True, SM, config=cfg)
        if n * k <= 300000:
            kernel_model.replay(n, k, p)


@pytest.mark.parametrize("G,dk,dv", [(1, 128, 128), (4, 64, 64), (16, 16, 64), (2, 256, 256), (8, 32, 32),
                                     (1, 64, 8), (32, 8, 8), (3, 64, 64)])
@pytest.mark.parametrize("partial", [False, True])
def test_gla_store_o_schedule(G, dk, dv, partial):
    """The GLA step's vectorised o epilogue writes each output of a round
    once and reads only its heads' partials, for full and short last rounds."""
    cpr = dv // 8
    RP = max(1, (256 // G) // cpr)
    nh = max(1, G - 1) if partial else G
    kernel_model.gla_store_o_schedule(nh, G, dv, RP)

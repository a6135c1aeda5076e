"""Bitwise checks of the CUDA path (closed forms and integer-valued inputs),
ragged tails, offset pointers, edge cases, error paths and determinism.

With B and a integer-valued in {-3..3} every fp32 partial sum is an integer
below 2^24, hence exact in any order: the output must then equal the
oracle's value rounded once to the output format, bit for bit, whatever the
variant, split or alignment.  That pins tails, split-K and the general
(realigning) variant exactly.
"""
from __future__ import annotations

import itertools
import os
import time

import numpy as np
import pytest
import torch

import memory_bound_gemv_02_gb300 as g
import oracle
from gpu_helpers import check_against_oracle, exact_bits_match, oracle_for, sample_rows
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu

CONFIGS = [None, {"variant": 2}, {"rows_per_warp": 4}, {"warps_per_cta": 4, "warp_split": 4},
           {"grid_split": 3}, {"grid_split": 2, "warp_split": 8}, {"ctas": 3},
           {"variant": 3}, {"variant": 3, "warp_split": 4}, {"variant": 3, "rows_per_warp": 4, "unroll": 2},
           {"variant": 3, "rows_per_warp": 2, "unroll": 4, "warps_per_cta": 8},
           {"variant": 3, "grid_split": 3, "warp_split": 2}, {"variant": 3, "ctas": 8},
           {"variant": 3, "l2_prefetch": 2}, {"variant": 3, "l2_prefetch": 1, "warp_split": 4, "overlap": 2},
           {"variant": 3, "warp_split": 4, "rows_per_warp": 2, "unroll": 4},
           {"variant": 3, "warp_split": 8, "rows_per_warp": 2, "unroll": 4},
           {"variant": 3, "warp_split": 2, "rows_per_warp": 2, "unroll": 4, "overlap": 2},
           {"variant": 4}, {"variant": 4, "stages": 2, "unroll": 4, "warp_split": 2},
           {"variant": 4, "grid_split": 3, "warps_per_cta": 8, "warp_split": 4, "overlap": 2}]


def _run(B, a, out_fp32=False, config=None, c=None):
    if config:
        return g.gemv_ex(B, a, c=c, out_fp32=out_fp32, config=config)
    return g.gemv(B, a, c=c, out_fp32=out_fp32)


def _run_valid(B, a, out_fp32=False, config=None, c=None):
    """As _run, but None when the forced configuration does not apply to
    this shape (e.g. several rows per warp with k % 8 != 0)."""
    try:
        return _run(B, a, out_fp32, config, c)
    except g.GemvError as e:
        assert e.status == g.GEMV_ERR_CONFIG
        return None


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("k", [1, 7, 8, 4096, 7169, 16384])
def test_ones_give_k(cuda_dev, dtype, k):
    B = torch.ones((37, k), dtype=inputs.TORCH_DTYPE[dtype], device=cuda_dev)
    a = torch.ones(k, dtype=B.dtype, device=cuda_dev)
    c32 = _run(B, a, True)
    assert (c32.cpu() == float(k)).all()  # exact in fp32
    c = _run(B, a, False)
    want = oracle.round_out(np.full(37, float(k)), dtype)
    assert (inputs.out_bits(c) == want).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(64, 100), (100, 64), (33, 33), (5, 4099)])
def test_identity_padded_gives_a(cuda_dev, dtype, n, k):
    B = torch.zeros((n, k), dtype=inputs.TORCH_DTYPE[dtype], device=cuda_dev)
    m = min(n, k)
    B[torch.arange(m), torch.arange(m)] = 1
    _, a = inputs.make_inputs(1, k, dtype, "uniform", 2, cuda_dev)
    for cfg in CONFIGS:
        c = _run_valid(B, a, False, cfg)
        if c is None:
            continue
        want = torch.zeros(n, dtype=B.dtype, device=cuda_dev)
        want[:m] = a[:m]
        assert (inputs.out_bits(c) == inputs.out_bits(want)).all(), cfg


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("out_fp32", [False, True])
@pytest.mark.parametrize("cfg", CONFIGS)
def test_integer_inputs_bit_exact(cuda_dev, dtype, out_fp32, cfg):
    for n, k in [(1, 1), (3, 9), (17, 31), (129, 257), (1000, 7169), (513, 4096), (64, 16384)]:
        B, a = inputs.make_int_inputs(n, k, dtype, seed=n + k, device=cuda_dev)
        c = _run_valid(B, a, out_fp32, cfg)
        if c is None:
            continue
        assert exact_bits_match(c, B, a, out_fp32), (n, k, cfg)


# Slices whose last step holds at most one block per lane (32 blocks) are
# folded into the step before; 33 blocks are not.  Row lengths (in 16-byte
# blocks) of 32*U*m + {1, 2, 32, 33} with U = 8 (steps of 256 blocks) and
# U = 4 (128), for one and two warps per row; k % 8 != 0 adds the edge block
# of unaligned rows.
FOLD_K = [1032, 1288, 2049, 2056, 2304, 2328, 4104, 4112, 4113]
FOLD_CONFIGS = [{"variant": 3, "warp_split": 1, "rows_per_warp": 1, "unroll": 8},
                {"variant": 3, "warp_split": 1, "rows_per_warp": 2, "unroll": 4},
                {"variant": 3, "warp_split": 2, "rows_per_warp": 1, "unroll": 8}]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("cfg", FOLD_CONFIGS)
def test_folded_last_step_bit_exact(cuda_dev, dtype, cfg):
    """The fold, and its boundary (a remainder of 33 blocks is a step of its
    own), in every launch mode (the second step's L2 prefetch differs between
    them) and at a B offset: integer inputs, so the output is bit-exact."""
    for k in FOLD_K:
        B, a = inputs.make_int_inputs(300, k, dtype, seed=k, device=cuda_dev)
        buf = torch.zeros(300 * k + 8, dtype=B.dtype, device=cuda_dev)
        Bo = buf[3:3 + 300 * k].view(300, k)
        Bo.copy_(B)
        for Bx in (B, Bo):
            for overlap in (0, 1, 2):
                c = _run_valid(Bx, a, False, {**cfg, "overlap": overlap})
                if c is None:
                    continue
                assert exact_bits_match(c, Bx, a, False), (k, cfg, overlap, Bx.data_ptr() % 16)


def test_benchmark_plan_bit_exact_full_size(cuda_dev):
    """The benchmark workload's shape in the plan gemv() picks for it (two
    rows per warp, four warps per pair of rows), with integer inputs: every
    row bit-exact, in both overlap modes the benchmark reports."""
    n, k = 7168, 16384
    B, a = inputs.make_int_inputs(n, k, "f16", seed=5, device=cuda_dev)
    plan = g.gemv_plan(n, k, g.GEMV_F16, True, torch.cuda.get_device_properties(cuda_dev).multi_processor_count)
    assert (plan["warp_split"], plan["rows_per_warp"], plan["unroll"]) == (4, 2, 4)
    for cfg in (None, {"overlap": 2}):
        c = _run(B, a, False, cfg)
        assert exact_bits_match(c, B, a, False), cfg


# Every n and k in 1..17, 31..33, 255..257, and 4099 and 7169 (paired with
# the small sizes: large x large is covered by the workload tests).
TAIL_N = list(range(1, 18)) + [31, 32, 33, 255, 256, 257, 4099, 7169]
TAIL_K = list(range(1, 18)) + [31, 32, 33, 255, 256, 257, 4099, 7169]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("variant", [None, 3, 4])
def test_ragged_tails_bit_exact(cuda_dev, dtype, variant):
    cfg = {"variant": variant} if variant else None
    for n, k in itertools.product(TAIL_N, TAIL_K):
        if n > 257 and k > 257:
            continue
        B, a = inputs.make_int_inputs(n, k, dtype, seed=7 * n + k, device=cuda_dev)
        c = _run(B, a, False, cfg)
        assert exact_bits_match(c, B, a, False), (n, k, cfg)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("b_off,a_off", [(1, 0), (0, 1), (3, 5), (7, 7)])
def test_offset_views_take_the_general_path(cuda_dev, dtype, b_off, a_off):
    """B and a starting at element offsets (not 16-byte aligned)."""
    td = inputs.TORCH_DTYPE[dtype]
    for n, k in [(50, 64), (33, 4096), (9, 7169)]:
        Bi, ai = inputs.make_int_inputs(n, k, dtype, seed=n, device=cuda_dev)
        Bbuf = torch.zeros(n * k + 16, dtype=td, device=cuda_dev)
        abuf = torch.zeros(k + 16, dtype=td, device=cuda_dev)
        Bv = Bbuf[b_off:b_off + n * k].view(n, k)
        av = abuf[a_off:a_off + k]
        Bv.copy_(Bi)
        av.copy_(ai)
        c = _run(Bv, av, False)
        if b_off % 8 or k % 8:
            assert g.gemv_last_config()["variant"] in (g.GEMV_VARIANT_ROWS_GENERAL, g.GEMV_VARIANT_TILES)
        assert exact_bits_match(c, Bi, ai, False), (n, k, b_off, a_off)
        c = _run(Bv, av, False, {"variant": 3})
        assert exact_bits_match(c, Bi, ai, False), (n, k, b_off, a_off, "tiles")
        c = _run(Bv, av, False, {"variant": 4})
        assert exact_bits_match(c, Bi, ai, False), (n, k, b_off, a_off, "bulk")
        Bu, au = inputs.make_inputs(n, k, dtype, "uniform", 9, cuda_dev)
        Bv.copy_(Bu)
        av.copy_(au)
        c = _run(Bv, av, True)
        check_against_oracle(c, Bu, au, True, label=f"offset {b_off},{a_off} {n}x{k}")


def test_output_guard_bands_untouched(cuda_dev):
    for out_fp32 in (False, True):
        for cfg in CONFIGS:
            B, a = inputs.make_inputs(1001, 3001, "bf16", "uniform", 4, cuda_dev)
            dt = torch.float32 if out_fp32 else torch.bfloat16
            buf = torch.full((1001 + 256,), 1234.5, dtype=dt, device=cuda_dev)
            c = buf[128:128 + 1001]
            if _run_valid(B, a, out_fp32, cfg, c=c) is None:
                continue
            torch.cuda.synchronize()
            assert (buf[:128] == 1234.5).all() and (buf[128 + 1001:] == 1234.5).all(), cfg
            check_against_oracle(c, B, a, out_fp32, label=f"guard {cfg}")


def test_empty_and_degenerate_sizes(cuda_dev):
    B = torch.empty((0, 64), dtype=torch.float16, device=cuda_dev)
    a = torch.ones(64, dtype=torch.float16, device=cuda_dev)
    assert g.gemv(B, a).numel() == 0
    B = torch.empty((5, 0), dtype=torch.bfloat16, device=cuda_dev)
    a = torch.empty(0, dtype=torch.bfloat16, device=cuda_dev)
    c = torch.full((5,), 7.0, dtype=torch.bfloat16, device=cuda_dev)
    g.gemv(B, a, c=c)
    torch.cuda.synchronize()
    assert (inputs.out_bits(c) == 0).all()  # +0: the empty sum


def test_nonfinite_inputs_stay_in_their_rows(cuda_dev):
    for dtype in ("f16", "bf16"):
        for k in (64, 67):
            B, a = inputs.make_int_inputs(8, k, dtype, seed=1, device=cuda_dev)
            B[2, 5] = float("inf")
            B[5, k - 1] = float("nan")
            B[6, 0] = float("-inf")
            for cfg in CONFIGS:
                c = _run_valid(B, a, True, cfg)
                if c is None:
                    continue
                c = c.cpu()
                want, _ = oracle_for(B, a)
                for i in range(8):
                    if np.isnan(want[i]):
                        assert torch.isnan(c[i]), (i, cfg)
                    else:
                        assert c[i].item() == want[i], (i, cfg, c[i].item(), want[i])


def test_error_paths_launch_nothing(cuda_dev):
    B, a = inputs.make_inputs(64, 128, "f16", "uniform", 0, cuda_dev)
    with pytest.raises(g.GemvError) as ei:
        g.gemv(B, a, c=B.view(-1)[:64])  # c inside B
    assert ei.value.status == g.GEMV_ERR_ALIAS
    with pytest.raises(g.GemvError) as ei:
        g.gemv_ex(B, a, config={"grid_split": 100000})  # more than 65536 k-segments
    assert ei.value.status == g.GEMV_ERR_CONFIG
    g.gemv_debug_inject(g.GEMV_ERR_CUDA)
    c = torch.full((64,), 3.0, dtype=torch.float16, device=cuda_dev)
    with pytest.raises(g.GemvError) as ei:
        g.gemv(B, a, c=c)
    assert ei.value.status == g.GEMV_ERR_CUDA
    torch.cuda.synchronize()
    assert (c == 3.0).all()  # nothing ran
    g.gemv(B, a, c=c)  # the injected status was one-shot; the context is healthy
    check_against_oracle(c, B, a, False)


def test_determinism_repeated_calls(cuda_dev):
    """Fixed-order reductions: 200 calls give bitwise-identical results (a
    race in the cross-warp or split-K combination would show up here)."""
    for cfg in (None, {"warp_split": 8, "warps_per_cta": 16}, {"grid_split": 4},
                {"variant": 3, "warp_split": 4}, {"variant": 3, "grid_split": 2, "warp_split": 8},
                {"variant": 4, "warp_split": 4}, {"variant": 4, "grid_split": 2, "warp_split": 8, "stages": 2}):
        B, a = inputs.make_inputs(3001, 5000, "f16", "normal", 2, cuda_dev, b_sigma=0.5)
        first = _run(B, a, True, cfg).clone()
        c = torch.empty_like(first)
        for _ in range(200):
            _run(B, a, True, cfg, c=c)
            assert torch.equal(c, first), cfg


def test_concurrent_streams_split_k(cuda_dev):
    """Split-K workspaces are per stream: concurrent calls do not interfere."""
    streams = [torch.cuda.Stream() for _ in range(3)]
    data = [inputs.make_inputs(333, 20000, "bf16", "uniform", s, cuda_dev) for s in range(3)]
    outs = []
    for s, (B, a) in zip(streams, data):
        with torch.cuda.stream(s):
            outs.append(g.gemv_ex(B, a, out_fp32=True, config={"grid_split": 4}, stream=s))
    torch.cuda.synchronize()
    for (B, a), c in zip(data, outs):
        check_against_oracle(c, B, a, True)


def test_gemv_host_end_to_end(cuda_dev):
    n, k = 1000, 3000
    Bd, ad = inputs.make_inputs(n, k, "f16", "uniform", 3, cuda_dev)
    Bh = Bd.cpu().pin_memory()
    ah = ad.cpu().pin_memory()
    ch = torch.empty(n, dtype=torch.float16).pin_memory()
    B_dev = torch.empty_like(Bd)
    a_dev = torch.empty_like(ad)
    c_dev = torch.empty(n, dtype=torch.float16, device=cuda_dev)
    g.gemv_host(Bh, ah, ch, B_dev, a_dev, c_dev)
    torch.cuda.synchronize()
    check_against_oracle(ch.to(cuda_dev), Bd, ad, False, label="gemv_host")


def test_host_overhead_per_call(cuda_dev):
    """A cached-key call costs microseconds of host time (the pages' Case B.4
    saw 11 ms per call from rebuilding a closure).  Measured on the raw
    C entry point with enqueue-only timing."""
    B, a = inputs.make_inputs(256, 512, "f16", "uniform", 0, cuda_dev)
    c = torch.empty(256, dtype=torch.float16, device=cuda_dev)
    L = g.lib()
    s = torch.cuda.current_stream().cuda_stream
    args = (B.data_ptr(), a.data_ptr(), c.data_ptr(), 256, 512, 0, s)
    assert L.gemv(*args) == 0
    torch.cuda.synchronize()
    per = []
    for _ in range(20):
        t0 = time.perf_counter()
        for _ in range(200):  # bursts short enough never to fill the launch queue
            L.gemv(*args)
        per.append((time.perf_counter() - t0) / 200)
        torch.cuda.synchronize()
    med = float(np.median(per))
    assert med < 10e-6, f"host time per call {med * 1e6:.2f} us"


@pytest.mark.parametrize("overlap", [1, 2])
@pytest.mark.parametrize("variant", [None, 3, 4])
def test_overlap_respects_dependencies(cuda_dev, overlap, variant):
    """Programmatic dependent launch: each call still sees the memory of the
    kernels before it.  A chain x_{m+1} = B @ x_m (c of one call is a of the
    next), torch kernels rewriting a between calls, and two calls writing the
    same c with different B."""
    cfg = {"overlap": overlap}
    if variant:
        cfg["variant"] = variant
    n = 2048
    B, x0 = inputs.make_int_inputs(n, n, "bf16", seed=3, device=cuda_dev, lo=-1, hi=1)
    B = B * (1.0 / 64)  # keeps the chain's values inside bf16 range, exactly
    xs = [x0]
    for _ in range(12):
        xs.append(g.gemv_ex(B, xs[-1], config=cfg))
    torch.cuda.synchronize()
    for m in range(12):
        check_against_oracle(xs[m + 1], B, xs[m], False, label=f"chain step {m} overlap {overlap}")
    # a rewritten by a torch kernel right before each call
    a = torch.empty(n, dtype=torch.bfloat16, device=cuda_dev)
    outs = []
    for m in range(6):
        a.copy_(xs[m])
        outs.append(g.gemv_ex(B, a, config=cfg))
    torch.cuda.synchronize()
    for m in range(6):
        check_against_oracle(outs[m], B, xs[m], False, label=f"a rewritten {m}")
    # same c written by consecutive calls: the last one wins
    B2 = B * 2
    c = torch.empty(n, dtype=torch.bfloat16, device=cuda_dev)
    for _ in range(5):
        g.gemv_ex(B, xs[0], c=c, config=cfg)
        g.gemv_ex(B2, xs[0], c=c, config=cfg)
    check_against_oracle(c, B2, xs[0], False, label="WAW on c")


@pytest.mark.parametrize("variant", [None, 3, 4])
def test_overlap_pdl_sees_rewritten_B(cuda_dev, variant):
    """GEMV_OVERLAP_PDL (without the B prefetch) also orders B: a kernel that
    rewrites B right before the call is waited for."""
    cfg = {"overlap": 1}
    if variant:
        cfg["variant"] = variant
    B, a = inputs.make_inputs(3000, 4104, "f16", "uniform", 6, cuda_dev)
    Bw = torch.empty_like(B)
    for m in range(4):
        Bw.copy_(B * (m + 1))
        c = g.gemv_ex(Bw, a, config=cfg)
        check_against_oracle(c, B * (m + 1), a, False, label=f"B rewritten {m}")


def test_overlap_uses_cached_plan(cuda_dev):
    B, a = inputs.make_inputs(777, 5000, "bf16", "uniform", 7, cuda_dev)
    g.gemv(B, a)
    base = g.gemv_last_config()
    assert base["overlap"] == g.GEMV_OVERLAP_PDL  # gemv() launches as a programmatic dependent launch
    g.gemv_ex(B, a, config={})
    assert g.gemv_last_config()["overlap"] == g.GEMV_OVERLAP_NONE  # a given configuration is taken as is
    g.gemv_ex(B, a, config={"overlap": 2})
    got = g.gemv_last_config()
    assert got["overlap"] == 2
    assert {k: v for k, v in got.items() if k != "overlap"} == {k: v for k, v in base.items() if k != "overlap"}
    with pytest.raises(g.GemvError) as ei:
        g.gemv_ex(B, a, config={"overlap": 4})
    assert ei.value.status == g.GEMV_ERR_CONFIG


@pytest.mark.parametrize("variant", [None, 3, 1, 4])
def test_overlap_prefetch_ba_shared_input(cuda_dev, variant):
    """GEMV_OVERLAP_PDL_PREFETCH_BA (B and a promised unwritten by the work in
    flight): several GEMVs on one input vector, e.g. the projections of one
    activation, including consecutive calls that write the same c."""
    cfg = {"overlap": 3}
    if variant:
        cfg["variant"] = variant
    n, k = 3000, 4104
    _, a = inputs.make_inputs(1, k, "bf16", "uniform", 8, cuda_dev)
    Bs = [inputs.make_inputs(n, k, "bf16", "uniform", 20 + i, cuda_dev)[0] for i in range(4)]
    outs = [g.gemv_ex(B, a, config=cfg) for B in Bs]
    c = torch.empty(n, dtype=torch.bfloat16, device=cuda_dev)
    for _ in range(3):
        for B in Bs:
            g.gemv_ex(B, a, c=c, config=cfg)
    torch.cuda.synchronize()
    for i, B in enumerate(Bs):
        check_against_oracle(outs[i], B, a, False, label=f"shared input, B{i}")
    check_against_oracle(c, Bs[-1], a, False, label="last writer of c")


def test_native_measurement_tool(cuda_dev):
    """The native (C++) measurements beside the benchmark: the host cost of a
    cached gemv() call is under 10 us and within a few microseconds of an
    empty kernel launch, and the read-only stream reaches a plausible
    fraction of the HBM bandwidth (above 3 TB/s, below the 8 TB/s nominal
    peak plus a margin for the timer)."""
    import json
    import subprocess

    from memory_bound_gemv_02_gb300 import _build
    assert os.path.exists(_build.HOST_TOOL), "the build makes the native measurement tool"
    r = subprocess.run([_build.HOST_TOOL], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert 0 < d["gemv_us"] < 10.0
    assert 0 < d["empty_launch_us"] <= d["gemv_us"] + 1.0
    for key in ("read_gbs_1gib_plain", "read_gbs_1gib_overlapped", "read_gbs_small_plain",
                "read_gbs_small_overlapped"):
        assert 3000.0 < d[key] < 8500.0, (key, d[key])


@pytest.mark.parametrize("n,k,dtype,cfg", [(2, 3_000_000, "f16", None), (3, 5_000_001, "bf16", None),
                                           (2, 3_000_000, "bf16", {"variant": 4}), (64, 2**22, "f16", None)])
def test_long_rows_against_oracle(cuda_dev, n, k, dtype, cfg):
    """Rows longer than 64 segments of 32768 columns (thousands of k-segments
    for the longest; the second pass then takes a warp per row)."""
    B, a = inputs.make_inputs(n, k, dtype, "uniform", 11, cuda_dev)
    for out_fp32 in (False, True):
        c = _run(B, a, out_fp32, cfg)
        check_against_oracle(c, B, a, out_fp32, label=f"{n}x{k} {dtype} {cfg} f32={out_fp32}")
    assert g.gemv_last_config()["grid_split"] > 64


def test_maximum_k_ones_closed_form(cuda_dev):
    """n = 1, k = INT32_MAX (4 GiB of B and of a): with B = a = ones every
    partial is exact, so the result is k rounded once -- 2^31 in fp32 and bf16,
    +inf in fp16 (beyond 65504) -- the closed form c_i = k."""
    k = 2**31 - 1
    B = torch.ones((1, k), dtype=torch.float16, device=cuda_dev)
    a = torch.ones(k, dtype=torch.float16, device=cuda_dev)
    c32 = _run(B, a, True)
    c16 = _run(B, a, False)
    torch.cuda.synchronize()
    assert g.gemv_last_config()["grid_split"] == 65536
    assert c32.item() == float(2**31)
    assert torch.isinf(c16).all() and c16.item() > 0
    del B, a
    Bb = torch.ones((1, k), dtype=torch.bfloat16, device=cuda_dev)
    ab = torch.ones(k, dtype=torch.bfloat16, device=cuda_dev)
    cb = _run(Bb, ab, False)
    torch.cuda.synchronize()
    assert (inputs.out_bits(cb) == oracle.round_out(np.array([float(k)]), "bf16")).all()


@pytest.mark.parametrize("n,k,dtype", [(3000, 4104, "bf16"), (1_400_000, 16, "f16"), (513, 7169, "f16"),
                                       (2048, 16384, "bf16")])
def test_shared_input_deferred_stores(cuda_dev, n, k, dtype):
    """GEMV_OVERLAP_PDL_PREFETCH_BA: the tiles kernel keeps its row results
    in shared memory and stores them after one wait (up to 4096 rows per
    CTA; beyond that, as 1.4M rows of 16 here, it stores as it goes).  A
    chain of calls sharing a, each writing the same c and then its own,
    all checked."""
    cfg = {"overlap": 3, "variant": 3}
    _, a = inputs.make_inputs(1, k, dtype, "uniform", 12, cuda_dev)
    Bs = [inputs.make_inputs(n, k, dtype, "uniform", 30 + i, cuda_dev)[0] for i in range(3)]
    c = torch.empty(n, dtype=Bs[0].dtype, device=cuda_dev)
    outs = []
    for _ in range(2):
        for B in Bs:
            g.gemv_ex(B, a, c=c, config=cfg)
            outs.append(g.gemv_ex(B, a, config=cfg))
    torch.cuda.synchronize()
    rows = sample_rows(n, 160)
    check_against_oracle(c, Bs[-1], a, False, rows=rows, label="last writer of c")
    for i, o in enumerate(outs[:3]):
        check_against_oracle(o, Bs[i], a, False, rows=rows, label=f"shared input B{i}")

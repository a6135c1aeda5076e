"""The bulk variant on the GPU: B staged in shared memory by 1-D bulk
asynchronous copies into per-warp mbarrier rings (the sm_103a form of the
multi-stage B pipeline of TileLang Case Studies, Case B.1 "O3 Pipelined B
Loads"), against the oracle.

Same tolerances as every GEMV path (16-bit output 1e-2 * max(1, |c_ref|),
fp32 output 1e-5 * sum |B a|, the power-of-two rule).  With equal warps per
CTA, warp split, unroll and k-segments, each lane of the bulk kernel visits
the same blocks in the same order as the tiles kernel with one row per warp,
and the warp and slice reductions are the same: the two must then agree bit
for bit.  The ring's error path (a wait that gives up) is exercised with a
zero poll budget, which hangs nothing: the copies complete, the kernel only
stops waiting for them.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import memory_bound_gemv_02_gb300 as g
from gpu_helpers import check_against_oracle, exact_bits_match, sample_rows
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu

BULK = [{"variant": 4}, {"variant": 4, "stages": 2}, {"variant": 4, "stages": 3, "unroll": 4},
        {"variant": 4, "unroll": 8, "stages": 2}, {"variant": 4, "warp_split": 2},
        {"variant": 4, "warps_per_cta": 8, "warp_split": 4, "stages": 3}, {"variant": 4, "grid_split": 3},
        {"variant": 4, "ctas": 8}, {"variant": 4, "warps_per_cta": 4, "warp_split": 2, "grid_split": 2, "stages": 5},
        {"variant": 4, "stages": 8, "unroll": 4}, {"variant": 4, "overlap": 2}, {"variant": 4, "overlap": 3}]

SHAPES = [(1, 1), (3, 9), (17, 7), (64, 512), (33, 1000), (9, 5000), (40, 4099), (5, 16384), (2, 33000),
          (300, 24), (130, 2056), (1031, 4099), (2048, 8192)]


def _bulk(B, a, out_fp32, cfg, c=None):
    try:
        return g.gemv_ex(B, a, c=c, out_fp32=out_fp32, config=cfg)
    except g.GemvError as e:
        assert e.status == g.GEMV_ERR_CONFIG
        return None


@pytest.mark.parametrize("cfg", BULK)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("out_fp32", [False, True])
def test_bulk_parity(cuda_dev, cfg, dtype, out_fp32):
    for n, k in SHAPES:
        B, a = inputs.make_inputs(n, k, dtype, "uniform", n + 3 * k, cuda_dev)
        c = _bulk(B, a, out_fp32, cfg)
        if c is None:
            continue
        assert g.gemv_last_config()["variant"] == g.GEMV_VARIANT_BULK
        check_against_oracle(c, B, a, out_fp32, label=f"bulk {n}x{k} {cfg}")


@pytest.mark.parametrize("cfg", BULK[:6])
@pytest.mark.parametrize("b_off", [0, 1, 5])
def test_bulk_integer_inputs_bit_exact(cuda_dev, cfg, b_off):
    """Integer inputs make every fp32 sum exact; B starts b_off elements
    into its buffer (every row offset class when k % 8 != 0)."""
    for n, k in [(1, 1), (17, 31), (129, 257), (1000, 7169), (64, 16384), (9, 5000)]:
        Bi, a = inputs.make_int_inputs(n, k, "bf16", seed=n + k + b_off, device=cuda_dev)
        buf = torch.zeros(n * k + 16, dtype=Bi.dtype, device=cuda_dev)
        Bv = buf[b_off:b_off + n * k].view(n, k)
        Bv.copy_(Bi)
        for out_fp32 in (False, True):
            c = _bulk(Bv, a, out_fp32, cfg)
            if c is None:
                continue
            assert exact_bits_match(c, Bi, a, out_fp32), (n, k, b_off, cfg)


@pytest.mark.parametrize("W,S,U,Sg", [(16, 1, 8, 1), (16, 2, 8, 1), (16, 4, 8, 1), (8, 2, 4, 1), (16, 4, 4, 2),
                                      (4, 1, 4, 3), (16, 8, 8, 1)])
@pytest.mark.parametrize("aligned", [True, False])
def test_bulk_matches_tiles_bitwise(cuda_dev, W, S, U, Sg, aligned):
    n, k = (3001, 8192) if aligned else (3001, 8195)
    B, a = inputs.make_inputs(n, k, "f16", "normal", 11, cuda_dev, b_sigma=0.5)
    common = {"warps_per_cta": W, "warp_split": S, "unroll": U, "rows_per_warp": 1, "grid_split": Sg}
    for out_fp32 in (False, True):
        t = g.gemv_ex(B, a, out_fp32=out_fp32, config={"variant": 3, **common})
        for stages in (2, 3):
            b = _bulk(B, a, out_fp32, {"variant": 4, "stages": stages, **common})
            if b is None:
                continue
            torch.cuda.synchronize()
            assert (inputs.out_bits(b) == inputs.out_bits(t)).all(), (W, S, U, Sg, stages, out_fp32)


@pytest.mark.parametrize("n,k,dtype,out_fp32", [(7168, 16384, "f16", False), (18432, 7168, "bf16", True),
                                                (28672, 8192, "bf16", False), (16384, 7169, "f16", True)])
def test_bulk_full_size_sampled(cuda_dev, n, k, dtype, out_fp32):
    """The workload shapes, with the planner's bulk configuration and the
    PDL + B-prefetch launch the benchmark uses, on sampled rows."""
    B, a = inputs.make_inputs(n, k, dtype, "normal", 1, cuda_dev)
    rows = sample_rows(n)
    for cfg in ({"variant": 4}, {"variant": 4, "overlap": 2}):
        c = g.gemv_ex(B, a, out_fp32=out_fp32, config=cfg)
        check_against_oracle(c, B, a, out_fp32, rows=rows, label=f"bulk full {n}x{k} {cfg}")


@pytest.mark.parametrize("n,k,pad", [(300, 1000, 8), (300, 1000, 3), (129, 4096, 1), (77, 7169, 7)])
def test_bulk_strided_with_epilogue(cuda_dev, n, k, pad):
    """Row stride ldb = k + pad with NaN padding, and the fused epilogue."""
    ldb = k + pad
    buf = torch.full((n, ldb), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    Bc, a = inputs.make_inputs(n, k, "bf16", "uniform", 4, cuda_dev)
    buf[:, :k] = Bc
    Bv = buf[:, :k]
    for cfg in ({"variant": 4}, {"variant": 4, "warp_split": 2, "stages": 2}, {"variant": 4, "grid_split": 2}):
        c = g.gemv_fused(Bv, a, out_fp32=True, config=cfg)
        check_against_oracle(c, Bc, a, True, label=f"bulk strided ldb={ldb} {cfg}")
        y = g.gemv_fused(Bv, a, out_fp32=True, alpha=2.0, activation="relu", config=cfg)
        torch.cuda.synchronize()
        want = torch.relu(2.0 * c)
        assert torch.allclose(y, want, rtol=2e-6, atol=0), cfg


def test_bulk_nonfinite_edges_are_redone(cuda_dev):
    """k % 8 != 0: the edge blocks of a row also hold neighbouring rows'
    elements; an Inf there must not reach this row (the masked redo)."""
    n, k = 64, 67
    for cfg in ({"variant": 4}, {"variant": 4, "warp_split": 2, "stages": 2}):
        B, a = inputs.make_int_inputs(n, k, "f16", seed=2, device=cuda_dev)
        B[10, 0] = float("inf")
        B[20, k - 1] = float("nan")
        c = g.gemv_ex(B, a, out_fp32=True, config=cfg).cpu().numpy()
        Bf = B.double().cpu().numpy()
        want = Bf @ a.double().cpu().numpy()
        for i in range(n):
            if np.isnan(want[i]) or np.isinf(want[i]):
                assert not np.isfinite(c[i]), (i, cfg)
            else:
                assert c[i] == want[i], (i, cfg, c[i], want[i])


def test_bulk_determinism(cuda_dev):
    B, a = inputs.make_inputs(3001, 5000, "f16", "normal", 2, cuda_dev, b_sigma=0.5)
    for cfg in ({"variant": 4, "warp_split": 4}, {"variant": 4, "grid_split": 2, "warp_split": 8, "stages": 2}):
        ref = inputs.out_bits(g.gemv_ex(B, a, config=cfg))
        for _ in range(100):
            c = g.gemv_ex(B, a, config=cfg)
        torch.cuda.synchronize()
        assert (inputs.out_bits(c) == ref).all(), cfg


def test_bulk_wait_budget_error_path(cuda_dev):
    """A zero poll budget makes every ring wait give up at once: the kernel
    drains its copies, writes NaN for its rows and counts the timeouts; the
    next call is unaffected."""
    B, a = inputs.make_inputs(1031, 4099, "bf16", "uniform", 5, cuda_dev)
    g.gemv_wait_timeouts(reset=True)
    assert g.gemv_wait_timeouts() == 0
    for cfg in ({"variant": 4}, {"variant": 4, "warp_split": 4, "stages": 2}):
        g.gemv_debug_wait_budget(0)
        c = g.gemv_ex(B, a, out_fp32=True, config=cfg)
        torch.cuda.synchronize()
        assert torch.isnan(c).all(), cfg
        got = g.gemv_wait_timeouts(reset=True)
        lc = g.gemv_last_config()
        # the copies still land, so every drain completes: the top bit stays clear
        assert not got & g.GEMV_DRAIN_TIMEOUT, (hex(got), cfg)
        assert 1 <= got <= lc["ctas"] * lc["warps_per_cta"], (got, cfg)
        c = g.gemv_ex(B, a, out_fp32=True, config=cfg)  # the budget was one-shot
        check_against_oracle(c, B, a, True, label=f"after the error path {cfg}")
        assert g.gemv_wait_timeouts() == 0
    # a budget that is large enough changes nothing
    g.gemv_debug_wait_budget(1 << 16)
    c = g.gemv_ex(B, a, out_fp32=True, config={"variant": 4})
    check_against_oracle(c, B, a, True, label="explicit budget")
    assert g.gemv_wait_timeouts() == 0
    with pytest.raises(g.GemvError):
        g.gemv_debug_wait_budget(-2)

"""Parity of the CUDA path with the oracle, element by element.

* Sizes the oracle finishes in seconds, spanning several CTAs, k-segments and
  ragged tails: every output row is compared.
* The workload shapes at full size, in the launch configuration gemv() picks
  (the one the benchmark times): sampled rows (first, last, seeded random)
  are compared one by one with the oracle.

Tolerances: 1e-2 * max(1, |c_ref|) for 16-bit output, 1e-5 * sum_j |B_ij a_j|
for fp32 output, and any power-of-two error of 2^-4 or more above one ulp is
a hard failure (tests/parity_rules.py).
"""
from __future__ import annotations

import itertools

import pytest
import torch

import memory_bound_gemv_02_gb300 as g
from gpu_helpers import check_against_oracle, sample_rows
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu


def _run(B, a, out_fp32=False, config=None):
    if config:
        return g.gemv_ex(B, a, out_fp32=out_fp32, config=config)
    return g.gemv(B, a, out_fp32=out_fp32)


# ------------------------------------------------------ whole-output parity --

def test_small_workload_full_output(cuda_dev):
    """n=256, k=512, fp16, uniform[-1,1] from seed 0: every row."""
    B, a = inputs.make_inputs(256, 512, "f16", "uniform", 0, cuda_dev)
    c = _run(B, a)
    check_against_oracle(c, B, a, False, label="256x512 f16")


MID_SHAPES = [(1000, 4099), (513, 7169), (2048, 2048), (300, 16384), (77, 1000), (4099, 1000),
              (1, 65536), (9, 40000), (3000, 264)]


@pytest.mark.parametrize("n,k", MID_SHAPES)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("out_fp32", [False, True])
def test_mid_shapes_full_output(cuda_dev, n, k, dtype, out_fp32):
    B, a = inputs.make_inputs(n, k, dtype, "uniform", 1, cuda_dev)
    c = _run(B, a, out_fp32)
    check_against_oracle(c, B, a, out_fp32, label=f"{n}x{k} {dtype} f32out={out_fp32}")


# ------------------------------------------------- full-size workload shapes --

def test_workload_7168x16384_f16(cuda_dev):
    B, a = inputs.make_inputs(7168, 16384, "f16", "normal", 0, cuda_dev, b_sigma=0.02, a_sigma=1.0)
    c = _run(B, a)
    check_against_oracle(c, B, a, False, rows=sample_rows(7168), label="7168x16384 f16")


@pytest.mark.parametrize("out_fp32", [False, True])
def test_workload_18432x7168_bf16(cuda_dev, out_fp32):
    B, a = inputs.make_inputs(18432, 7168, "bf16", "normal", 0, cuda_dev, b_sigma=0.02, a_sigma=1.0)
    c = _run(B, a, out_fp32)
    check_against_oracle(c, B, a, out_fp32, rows=sample_rows(18432), label=f"18432x7168 bf16 {out_fp32}")


@pytest.mark.parametrize("n,k", [(4096, 4096), (14336, 4096), (4096, 14336), (28672, 8192)])
def test_workload_decode_set_bf16(cuda_dev, n, k):
    B, a = inputs.make_inputs(n, k, "bf16", "normal", 0, cuda_dev, b_sigma=0.02, a_sigma=1.0)
    c = _run(B, a)
    check_against_oracle(c, B, a, False, rows=sample_rows(n), label=f"{n}x{k} bf16")


SWEEP = list(itertools.product([1024, 4099, 18433, 65536], [1000, 4096, 7169, 16384]))


@pytest.mark.parametrize("n,k", SWEEP)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_workload_sweep(cuda_dev, n, k, dtype):
    """Bandwidth/tail sweep, uniform[-1,1] inputs from seeds 0-3."""
    for seed in range(4):
        B, a = inputs.make_inputs(n, k, dtype, "uniform", seed, cuda_dev)
        c = _run(B, a)
        check_against_oracle(c, B, a, False, rows=sample_rows(n, 96, seed),
                             label=f"{n}x{k} {dtype} seed {seed}")
        del B, a, c


def test_extended_production_shape(cuda_dev):
    """(57344, 7168), the largest production shape of Case B.3."""
    for dtype in ("f16", "bf16"):
        B, a = inputs.make_inputs(57344, 7168, dtype, "normal", 0, cuda_dev)
        c = _run(B, a)
        check_against_oracle(c, B, a, False, rows=sample_rows(57344, 128), label=f"57344x7168 {dtype}")
        del B, a, c


# --------------------------------------------------------- forced variants --

FORCED = [
    {"variant": 2},
    {"rows_per_warp": 2}, {"rows_per_warp": 4},
    {"warps_per_cta": 4}, {"warps_per_cta": 8, "warp_split": 8},
    {"warps_per_cta": 16, "warp_split": 4},
    {"grid_split": 2}, {"grid_split": 5, "warp_split": 2},
    {"ctas": 1}, {"ctas": 37, "rows_per_warp": 2},
    {"variant": 3}, {"variant": 3, "warp_split": 8}, {"variant": 3, "warp_split": 2, "warps_per_cta": 4},
    {"variant": 3, "rows_per_warp": 2, "unroll": 4}, {"variant": 3, "grid_split": 4},
    {"variant": 3, "l2_prefetch": 1}, {"variant": 3, "l2_prefetch": 3, "warp_split": 2},
    {"variant": 3, "l2_prefetch": 2, "rows_per_warp": 4, "unroll": 2, "overlap": 2},
]


@pytest.mark.parametrize("cfg", FORCED)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_forced_configs_parity(cuda_dev, cfg, dtype):
    B, a = inputs.make_inputs(1537, 4096, dtype, "normal", 3, cuda_dev, b_sigma=0.05)
    for out_fp32 in (False, True):
        c = _run(B, a, out_fp32, cfg)
        used = g.gemv_last_config()
        for key, v in cfg.items():
            if key not in ("ctas", "grid_split"):
                assert used[key] == v, key
        check_against_oracle(c, B, a, out_fp32, label=f"{cfg} {dtype} f32out={out_fp32}")


def test_errors_differ_across_variants(cuda_dev):
    """Case A's rule: a design-level bug shows one identical error across
    every configuration.  Distinct launch configurations sum in distinct
    orders, so their fp32-output errors must not all coincide."""
    B, a = inputs.make_inputs(2048, 8192, "bf16", "uniform", 5, cuda_dev)
    import gpu_helpers as h
    c_ref, _ = h.oracle_for(B, a)
    maxerrs = set()
    for cfg in [None, {"rows_per_warp": 2}, {"warp_split": 4, "warps_per_cta": 16}, {"grid_split": 3},
                {"variant": 2}, {"variant": 3}]:
        c = _run(B, a, True, cfg)
        torch.cuda.synchronize()
        err = abs(h.gpu_values(c) - c_ref).max()
        maxerrs.add(float(err))
    assert len(maxerrs) >= 2


@pytest.mark.parametrize("n,k,dtype", [(7168, 16384, "f16"), (18432, 7168, "bf16"), (65536, 7169, "f16"),
                                       (18433, 7169, "bf16"), (4099, 1000, "f16"), (1024, 16384, "bf16"),
                                       (256, 512, "f16")])
def test_tiles_variant_workloads(cuda_dev, n, k, dtype):
    B, a = inputs.make_inputs(n, k, dtype, "uniform", 1, cuda_dev)
    for out_fp32 in (False, True):
        c = _run(B, a, out_fp32, {"variant": 3})
        check_against_oracle(c, B, a, out_fp32, rows=sample_rows(n, 128),
                             label=f"tiles {n}x{k} {dtype} f32out={out_fp32}")

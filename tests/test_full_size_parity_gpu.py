"""Every output row at full size, for every workload shape with n*k >= 1e8,
in the launch configuration gemv() picks (the one the benchmark times), one
seed each, against the oracle; and, with integer-valued inputs (every fp32
partial sum exact, so any summation order gives the same fp32 total), the
automatic plans of the largest shapes (the bulk kernel's) and an unaligned
tiles plan bit for bit, and the tiles kernel forced on the shapes the bulk
kernel serves.

The oracle runs over row chunks on a pool of host threads (rows are
independent; each chunk is one unchanged oracle call).
Tolerances as elsewhere: 1e-2 * max(1, |c_ref|) for 16-bit output,
1e-5 * sum_j |B_ij a_j| for fp32 output, power-of-two errors a hard failure.
"""
from __future__ import annotations

import pytest
import torch

import memory_bound_gemv_02_gb300 as g
from gpu_helpers import check_against_oracle, exact_bits_match
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu

# (n, k, dtype, fp32 output, distribution): the benchmark shape, the bf16
# shape in both output modes, the largest decode-set shape, the extended
# production shape, and the sweep members with n*k >= 1e8.
FULL = ([(7168, 16384, "f16", False, "normal"), (18432, 7168, "bf16", False, "normal"),
         (18432, 7168, "bf16", True, "normal"), (28672, 8192, "bf16", False, "normal"),
         (57344, 7168, "f16", False, "normal"), (57344, 7168, "bf16", False, "normal")]
        + [(n, k, dt, False, "uniform") for n, k in ((18433, 7169), (18433, 16384), (65536, 4096),
                                                      (65536, 7169), (65536, 16384)) for dt in ("f16", "bf16")])


@pytest.mark.parametrize("n,k,dtype,out_fp32,dist", FULL)
def test_every_row_at_full_size(cuda_dev, n, k, dtype, out_fp32, dist):
    assert n * k >= 10 ** 8
    B, a = inputs.make_inputs(n, k, dtype, dist, 0, cuda_dev)
    c = g.gemv(B, a, out_fp32=out_fp32)
    used = g.gemv_last_config()
    check_against_oracle(c, B, a, out_fp32, label=f"{n}x{k} {dtype} f32out={out_fp32} plan {used}")


# (n, k, dtype, the variant gemv() is expected to pick)
EXACT = [(57344, 7168, "f16", g.GEMV_VARIANT_BULK), (65536, 7169, "bf16", g.GEMV_VARIANT_BULK),
         (18433, 7169, "f16", g.GEMV_VARIANT_TILES), (18433, 16384, "bf16", g.GEMV_VARIANT_TILES)]


@pytest.mark.parametrize("n,k,dtype,variant", EXACT)
def test_automatic_plans_bit_exact_at_full_size(cuda_dev, n, k, dtype, variant):
    B, a = inputs.make_int_inputs(n, k, dtype, seed=n + k, device=cuda_dev)
    for out_fp32 in (False, True):
        c = g.gemv(B, a, out_fp32=out_fp32)
        used = g.gemv_last_config()
        assert used["variant"] == variant, used
        assert exact_bits_match(c, B, a, out_fp32), (n, k, dtype, out_fp32, used)
        del c
        torch.cuda.empty_cache()


@pytest.mark.parametrize("n,k,dtype", [(57344, 7168, "f16"), (65536, 7169, "bf16")])
def test_forced_tiles_plans_bit_exact_at_full_size(cuda_dev, n, k, dtype):
    """The tiles kernel (forced) on the large shapes the bulk kernel serves
    by default, its own plan, every row bit for bit with integer-valued
    inputs."""
    B, a = inputs.make_int_inputs(n, k, dtype, seed=n + k + 1, device=cuda_dev)
    for out_fp32 in (False, True):
        c = g.gemv_ex(B, a, out_fp32=out_fp32, config={"variant": g.GEMV_VARIANT_TILES})
        used = g.gemv_last_config()
        assert used["variant"] == g.GEMV_VARIANT_TILES, used
        assert exact_bits_match(c, B, a, out_fp32), (n, k, dtype, out_fp32, used)
        del c
        torch.cuda.empty_cache()

"""The row partition of one GEMV across replicas, through the library.

A multi-GPU run would give each rank a contiguous block of B's rows and a
copy of a; each rank's gemv() then produces its block of c, and nothing else
is exchanged.  Here the shards run one after another on the one GPU (no
shard waits on another): each shard's result must match the oracle on its
rows, the gathered c must match the oracle on every row, and with integer
inputs every shard is bit-exact whatever plan its row count gets.
"""
from __future__ import annotations

import pytest
import torch

import memory_bound_gemv_02_gb300 as g
from gpu_helpers import check_against_oracle, exact_bits_match
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu


def _shards(n, world):
    q, rem = divmod(n, world)
    out, r0 = [], 0
    for rank in range(world):
        r1 = r0 + q + (1 if rank < rem else 0)
        out.append((r0, r1))
        r0 = r1
    return out


@pytest.mark.parametrize("world", [2, 4, 8])
@pytest.mark.parametrize("n,k,dtype", [(18432, 7168, "bf16"), (7168, 16384, "f16"), (1031, 4099, "f16")])
def test_row_shards_gather_to_the_full_result(cuda_dev, world, n, k, dtype):
    B, a = inputs.make_inputs(n, k, dtype, "normal", 0, cuda_dev)
    c = torch.empty(n, dtype=B.dtype, device=cuda_dev)
    for r0, r1 in _shards(n, world):
        g.gemv(B[r0:r1], a, c=c[r0:r1])  # this rank's rows, a replicated
    check_against_oracle(c, B, a, False, label=f"{world} shards of {n}x{k} {dtype}")


@pytest.mark.parametrize("world", [3, 8])
def test_row_shards_bit_exact(cuda_dev, world):
    n, k = 4099, 7169
    B, a = inputs.make_int_inputs(n, k, "bf16", seed=9, device=cuda_dev)
    c = torch.empty(n, dtype=torch.float32, device=cuda_dev)
    for r0, r1 in _shards(n, world):
        g.gemv(B[r0:r1], a, c=c[r0:r1], out_fp32=True)
    assert exact_bits_match(c, B, a, True)

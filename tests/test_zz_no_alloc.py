"""The allocation-free split-K entry point, called through the C ABI.

Some callers cannot allocate device memory while they run -- an inference
engine's plugin code that is forbidden to call cudaMalloc during execution, a
serving loop where a cudaMalloc would synchronize the device and stall the
other streams, a process whose device memory is handed out up front by its
own allocator.  gemv_splitk_noalloc() keeps its split-K partial sums in a
fixed device array of the library instead of allocated memory.  Its output
must match the existing gemv() entry point's within the tolerances the other
tests use (1e-2 * max(1, |c|) for 16-bit output, 1e-5 * sum_j |B_ij a_j| for
fp32 output), on two calls in a row, and it must refuse, without launching, a
call whose partials would not fit in the array.

The file name makes pytest collect it last, so that a run stopping at the
first failure has already run every other test; it also passes alone in a
fresh process (its first call sets the scratch address up).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import memory_bound_gemv_02_gb300 as g
from gpu_helpers import check_against_oracle, oracle_for
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu


def _noalloc(B, a, c, out_fp32, grid_split):
    """Raw C-ABI call; returns the status code."""
    n, k = B.shape
    return g.lib().gemv_splitk_noalloc(B.data_ptr(), a.data_ptr(), c.data_ptr(), n, k,
                                       g.dtype_code(B.dtype, out_fp32), grid_split,
                                       torch.cuda.current_stream().cuda_stream)


def _matches_gemv(c_new, B, a, out_fp32, label):
    """Compare with gemv() on the same inputs, within the shared tolerances."""
    c_ref = g.gemv(B, a, out_fp32=out_fp32)
    torch.cuda.synchronize()
    x = c_new.double().cpu().numpy()
    y = c_ref.double().cpu().numpy()
    if out_fp32:
        _, s = oracle_for(B, a)
        tol = 1e-5 * s
    else:
        tol = 1e-2 * np.maximum(1.0, np.abs(y))
    bad = ~(np.abs(x - y) <= tol)
    assert not bad.any(), f"{label}: {int(bad.sum())} rows differ from gemv(), first {np.flatnonzero(bad)[:5]}"


CASES = [
    (64, 16384, "f16", False, 4),
    (300, 7169, "bf16", False, 3),
    (1024, 4096, "bf16", True, 2),
    (17, 65536, "f16", True, 8),
    (4099, 1000, "f16", False, 2),
]


@pytest.mark.parametrize("n,k,dtype,out_fp32,grid_split", CASES)
def test_two_calls_in_a_row_match_gemv(cuda_dev, n, k, dtype, out_fp32, grid_split):
    B1, a1 = inputs.make_inputs(n, k, dtype, "uniform", 11, cuda_dev)
    B2, a2 = inputs.make_inputs(n, k, dtype, "normal", 12, cuda_dev, b_sigma=0.5)
    odt = torch.float32 if out_fp32 else B1.dtype
    c1 = torch.full((n,), 7.0, dtype=odt, device=cuda_dev)
    c2 = torch.full((n,), 7.0, dtype=odt, device=cuda_dev)
    # two calls back to back on one stream: the second reuses the scratch
    assert _noalloc(B1, a1, c1, out_fp32, grid_split) == g.GEMV_OK
    assert _noalloc(B2, a2, c2, out_fp32, grid_split) == g.GEMV_OK
    torch.cuda.synchronize()
    _matches_gemv(c1, B1, a1, out_fp32, f"first call {n}x{k}")
    _matches_gemv(c2, B2, a2, out_fp32, f"second call {n}x{k}")
    check_against_oracle(c2, B2, a2, out_fp32, label=f"noalloc vs oracle {n}x{k}")


def test_offset_B_and_ragged_k(cuda_dev):
    n, k = 129, 7169
    Bi, ai = inputs.make_inputs(n, k, "bf16", "uniform", 4, cuda_dev)
    buf = torch.zeros(n * k + 8, dtype=torch.bfloat16, device=cuda_dev)
    Bv = buf[3:3 + n * k].view(n, k)
    Bv.copy_(Bi)
    for _ in range(2):
        c = torch.empty(n, dtype=torch.bfloat16, device=cuda_dev)
        assert _noalloc(Bv, ai, c, False, 5) == g.GEMV_OK
        torch.cuda.synchronize()
        _matches_gemv(c, Bi, ai, False, "offset B")


def test_oversized_call_is_refused_without_launching(cuda_dev):
    n = g.GEMV_STATIC_SCRATCH_FLOATS // 2 + 1  # 2 segments need one float too many
    k = 64
    B, a = inputs.make_inputs(n, k, "f16", "uniform", 1, cuda_dev)
    c = torch.full((n,), 3.0, dtype=torch.float16, device=cuda_dev)
    assert _noalloc(B, a, c, False, 2) == g.GEMV_ERR_SCRATCH
    torch.cuda.synchronize()
    assert (c == 3.0).all()
    assert _noalloc(B, a, c, False, 1) == g.GEMV_ERR_CONFIG  # split-K needs >= 2 segments
    # one segment fewer rows fits
    n2 = g.GEMV_STATIC_SCRATCH_FLOATS // 2
    c2 = torch.empty(n2, dtype=torch.float16, device=cuda_dev)
    assert _noalloc(B[:n2], a, c2, False, 2) == g.GEMV_OK
    torch.cuda.synchronize()
    _matches_gemv(c2, B[:n2], a, False, "largest fitting call")

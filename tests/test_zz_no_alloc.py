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
call whose partials would not fit in the array.  A call whose plan keeps a
single segment (k <= 8) writes c directly and needs no scratch however many
rows it has; a row longer than the requested split can stage takes more
segments.  And the call must not allocate: free device memory stays the same
across calls on streams the library has never seen, while the allocating
split-K path of gemv_ex() on such a stream visibly takes its workspace.

The file name makes pytest collect it last, so that a run stopping at the
first failure has already run every other test; it also passes alone in a
fresh process (its first call sets the scratch address up).
"""
from __future__ import annotations

import ctypes

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


def test_single_segment_needs_no_scratch(cuda_dev):
    # k = 8 leaves one segment whatever split is asked for: c is written
    # directly, so more rows than the scratch holds floats are fine
    n, k = g.GEMV_STATIC_SCRATCH_FLOATS + 1, 8
    B, a = inputs.make_inputs(n, k, "f16", "uniform", 5, cuda_dev)
    for out_fp32 in (False, True):
        c = torch.full((n,), 9.0, dtype=torch.float32 if out_fp32 else torch.float16, device=cuda_dev)
        assert _noalloc(B, a, c, out_fp32, 4) == g.GEMV_OK
        torch.cuda.synchronize()
        assert g.gemv_last_config()["grid_split"] == 1
        check_against_oracle(c, B, a, out_fp32, label=f"one segment, {n} rows")
        _matches_gemv(c, B, a, out_fp32, "one segment")


def test_long_rows_take_the_segments_they_need(cuda_dev):
    # 3 * 32768 + 5 columns need 4 segments of at most 32768; a split of 2
    # is raised to that
    n, k = 6, 3 * 32768 + 5
    B, a = inputs.make_inputs(n, k, "bf16", "uniform", 6, cuda_dev)
    for _ in range(2):
        c = torch.empty(n, dtype=torch.float32, device=cuda_dev)
        assert _noalloc(B, a, c, True, 2) == g.GEMV_OK
        torch.cuda.synchronize()
        assert g.gemv_last_config()["grid_split"] == 4
        check_against_oracle(c, B, a, True, label="long rows")
        _matches_gemv(c, B, a, True, "long rows")


def test_no_device_memory_is_allocated(cuda_dev):
    """Free device memory (cudaMemGetInfo) is unchanged across calls on a
    stream the library has never seen; as a control, the allocating split-K
    path (gemv_ex with the same split) on another new stream takes its
    workspace of grid_split * n floats (4 MiB here) and free memory drops."""
    n, k, split = 65536, 4096, 16  # 16 * 65536 floats: the whole scratch array
    B, a = inputs.make_inputs(n, k, "f16", "uniform", 7, cuda_dev)
    c = torch.empty(n, dtype=torch.float16, device=cuda_dev)
    c_ctl = torch.empty(n, dtype=torch.float16, device=cuda_dev)
    # The first call on the device looks the scratch address up and loads
    # the kernels (lazy module loading maps their code into device memory).
    assert _noalloc(B, a, c, False, split) == g.GEMV_OK
    torch.cuda.synchronize()
    s_new, s_ctl = torch.cuda.Stream(), torch.cuda.Stream()
    for st in (s_new, s_ctl):  # one ordinary launch on each new stream first
        with torch.cuda.stream(st):
            c.zero_()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    L = g.lib()
    for _ in range(3):
        assert L.gemv_splitk_noalloc(B.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, g.GEMV_F16, split,
                                     s_new.cuda_stream) == g.GEMV_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes across allocation-free calls"
    cfg = g.GemvConfig()
    cfg.variant = g.GEMV_VARIANT_TILES
    cfg.grid_split = split
    cfg.overlap = g.GEMV_OVERLAP_NONE
    assert L.gemv_ex(B.data_ptr(), a.data_ptr(), c_ctl.data_ptr(), n, k, g.GEMV_F16, ctypes.byref(cfg),
                     s_ctl.cuda_stream) == g.GEMV_OK
    torch.cuda.synchronize()
    free2, _ = torch.cuda.mem_get_info()
    assert free0 - free2 >= split * n * 4, "control: the allocating path's workspace should show"
    # (checked only now: copying c to the host allocates through torch)
    assert torch.equal(c_ctl, c)  # same plan, same kernels: bit-identical
    check_against_oracle(c, B, a, False, label="calls on a new stream")

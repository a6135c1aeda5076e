"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/gemv.h declares, and rejects bad arguments before touching
CUDA (on a machine without a GPU, a valid call reports GEMV_ERR_DEVICE)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gemv.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:gemv|gla)_?\w*)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_entry_points(gemv_lib):
    decl = _declared_functions()
    assert decl == sorted(gemv_lib.ENTRY_POINTS)


def test_library_exports_every_declared_symbol(gemv_lib):
    L = gemv_lib.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_status_strings(gemv_lib):
    for code in range(-9, 1):
        s = gemv_lib.gemv_status_string(code)
        assert s and s != "unknown status"
    assert gemv_lib.gemv_status_string(-99) == "unknown status"


# Fake, never-dereferenced addresses: validation is pure arithmetic.
B_ADDR, A_ADDR, C_ADDR = 0x7F0000000000, 0x7F1000000000, 0x7F2000000000


def _call(L, B, a, c, n, k, dtype):
    return L.gemv(B, a, c, n, k, dtype, None)


def test_argument_validation_without_gpu(gemv_lib):
    L = gemv_lib.lib()
    g = gemv_lib
    assert _call(L, B_ADDR, A_ADDR, C_ADDR, 4, 8, 7) == g.GEMV_ERR_DTYPE
    assert _call(L, B_ADDR, A_ADDR, C_ADDR, -1, 8, 0) == g.GEMV_ERR_ARG
    assert _call(L, B_ADDR, A_ADDR, C_ADDR, 4, -8, 0) == g.GEMV_ERR_ARG
    assert _call(L, B_ADDR, A_ADDR, C_ADDR, 4, 2 ** 31, 0) == g.GEMV_ERR_ARG
    assert _call(L, B_ADDR, A_ADDR, None, 4, 8, 0) == g.GEMV_ERR_ARG
    assert _call(L, None, A_ADDR, C_ADDR, 4, 8, 0) == g.GEMV_ERR_ARG
    assert _call(L, B_ADDR, None, C_ADDR, 4, 8, 0) == g.GEMV_ERR_ARG
    # n == 0 is a no-op that succeeds without any CUDA call
    assert _call(L, None, None, None, 0, 8, 0) == g.GEMV_OK
    # misaligned element pointers
    assert _call(L, B_ADDR + 1, A_ADDR, C_ADDR, 4, 8, 0) == g.GEMV_ERR_ALIGN
    assert _call(L, B_ADDR, A_ADDR + 1, C_ADDR, 4, 8, 0) == g.GEMV_ERR_ALIGN
    assert _call(L, B_ADDR, A_ADDR, C_ADDR + 2, 4, 8, g.GEMV_F16_OUT_F32) == g.GEMV_ERR_ALIGN
    # c overlapping B (B spans 4*8*2 = 64 bytes) or a
    assert _call(L, B_ADDR, A_ADDR, B_ADDR + 62, 4, 8, 0) == g.GEMV_ERR_ALIAS
    assert _call(L, B_ADDR, A_ADDR, A_ADDR - 6, 4, 8, 0) == g.GEMV_ERR_ALIAS
    assert _call(L, B_ADDR, A_ADDR, B_ADDR + 64, 4, 8, 0) != g.GEMV_ERR_ALIAS


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_reports_device_error(gemv_lib):
    L = gemv_lib.lib()
    assert _call(L, B_ADDR, A_ADDR, C_ADDR, 4, 8, 0) == gemv_lib.GEMV_ERR_DEVICE
    assert L.gemv_prepare(4, 8, 0, 1, None) == gemv_lib.GEMV_ERR_DEVICE


def test_debug_inject_is_one_shot(gemv_lib):
    L = gemv_lib.lib()
    gemv_lib.gemv_debug_inject(gemv_lib.GEMV_ERR_CUDA)
    assert _call(L, B_ADDR, A_ADDR, C_ADDR, 4, 8, 0) == gemv_lib.GEMV_ERR_CUDA
    # consumed: the next call is validated normally
    assert _call(L, B_ADDR, A_ADDR, C_ADDR, 4, 8, 9) == gemv_lib.GEMV_ERR_DTYPE
    gemv_lib.gemv_debug_inject(gemv_lib.GEMV_ERR_NOMEM)
    assert L.gemv_host(B_ADDR, A_ADDR, C_ADDR, B_ADDR, A_ADDR, C_ADDR, 4, 8, 0, None) == \
        gemv_lib.GEMV_ERR_NOMEM


def test_config_struct_layout_matches_header(gemv_lib):
    # int32 x 8, int64, int32 x 2, int32[4]  ->  8*4 + 8 + 2*4 + 16 = 64 bytes
    assert ctypes.sizeof(gemv_lib.GemvConfig) == 64
    assert gemv_lib.GemvConfig.k_segment.offset == 32


def test_fused_argument_validation_without_gpu(gemv_lib):
    L = gemv_lib.lib()
    g = gemv_lib
    ep = g.GemvEpilogue()
    ep.alpha, ep.beta = 1.0, 1.0
    call = lambda B, ldb, a, c, n, k, dt, e: L.gemv_fused(B, ldb, a, c, n, k, dt, e, None, None)
    assert call(B_ADDR, 7, A_ADDR, C_ADDR, 4, 8, 0, None) == g.GEMV_ERR_ARG      # ldb < k
    ep.activation = 9
    assert call(B_ADDR, 8, A_ADDR, C_ADDR, 4, 8, 0, ctypes.byref(ep)) == g.GEMV_ERR_ARG
    ep.activation = g.GEMV_ACT_SILU
    ep.bias_dtype = 5
    assert call(B_ADDR, 8, A_ADDR, C_ADDR, 4, 8, 0, ctypes.byref(ep)) == g.GEMV_ERR_ARG
    ep.bias_dtype = g.GEMV_BIAS_F32
    ep.bias = C_ADDR + 0x1002  # fp32 bias must be 4-byte aligned
    assert call(B_ADDR, 8, A_ADDR, C_ADDR, 4, 8, 0, ctypes.byref(ep)) == g.GEMV_ERR_ALIGN
    ep.bias = C_ADDR + 4  # overlaps c (4 fp16 outputs = 8 bytes)
    assert call(B_ADDR, 8, A_ADDR, C_ADDR, 4, 8, 0, ctypes.byref(ep)) == g.GEMV_ERR_ALIAS
    # c inside a padded B: rows of 8 elements with stride 64 span (3*64 + 8) * 2 bytes
    assert call(B_ADDR, 64, A_ADDR, B_ADDR + 300, 4, 8, 0, None) == g.GEMV_ERR_ALIAS
    assert call(B_ADDR, 64, A_ADDR, B_ADDR + 400, 4, 8, 0, None) != g.GEMV_ERR_ALIAS

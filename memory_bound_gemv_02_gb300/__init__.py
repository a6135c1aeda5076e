"""GB300-native GEMV ``c = B @ a`` -- thin Python binding of the C-ABI library.

B is (n, k) row-major, a is (k,), both fp16 or both bf16; products and sums in
fp32; c in the input type or fp32 (TileLang Case Studies, Case B
"Background").  Every step of the computation runs in the CUDA kernels of
``_lib/libgemv.so`` (sources in ``csrc/``, ABI in ``include/gemv.h``); this
module only marshals torch tensors into pointers, sizes and the current
stream.  There is no CPU or PyTorch fallback: if the library has not been
built, every call raises.

Names follow the C entry points: ``gemv``, ``gemv_ex``, ``gemv_fused``, ``gemv_prepare``,
``gemv_plan``, ``gemv_last_config``, ``gemv_status_string``,
``gemv_last_cuda_error``, ``gemv_debug_inject``, ``gemv_release``,
``gemv_host``, ``gemv_splitk_noalloc``, ``gemv_wait_timeouts``,
``gemv_debug_wait_budget``, ``gla_decode``, ``gla_decode_ex``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

GEMV_F16, GEMV_BF16, GEMV_F16_OUT_F32, GEMV_BF16_OUT_F32 = 0, 1, 2, 3
GEMV_OK = 0
GEMV_ERR_ARG, GEMV_ERR_DTYPE, GEMV_ERR_ALIAS, GEMV_ERR_DEVICE = -1, -2, -3, -4
GEMV_ERR_CUDA, GEMV_ERR_CONFIG, GEMV_ERR_ALIGN, GEMV_ERR_NOMEM = -5, -6, -7, -8
GEMV_ERR_SCRATCH = -9
GEMV_STATIC_SCRATCH_FLOATS = 1 << 20
GEMV_DRAIN_TIMEOUT = 0x80000000  # bit of gemv_wait_timeouts(): a drain of issued copies ran out
GEMV_VARIANT_AUTO, GEMV_VARIANT_ROWS, GEMV_VARIANT_ROWS_GENERAL, GEMV_VARIANT_TILES = 0, 1, 2, 3
GEMV_VARIANT_BULK = 4
GEMV_OVERLAP_NONE, GEMV_OVERLAP_PDL, GEMV_OVERLAP_PDL_PREFETCH_B, GEMV_OVERLAP_PDL_PREFETCH_BA = 0, 1, 2, 3
GEMV_ACT_NONE, GEMV_ACT_RELU, GEMV_ACT_SIGMOID, GEMV_ACT_SILU = 0, 1, 2, 3
GEMV_BIAS_INPUT_TYPE, GEMV_BIAS_F32 = 0, 1
GLA_F16, GLA_BF16, GLA_F32 = 0, 1, 2
GLA_VARIANT_AUTO, GLA_VARIANT_CTA, GLA_VARIANT_WARP, GLA_VARIANT_PIPE = 0, 1, 2, 3
GLA_PREFETCH_STATE = 1
_GLA_DTYPE = {torch.float16: GLA_F16, torch.bfloat16: GLA_BF16, torch.float32: GLA_F32}
ACTIVATIONS = {"none": GEMV_ACT_NONE, "relu": GEMV_ACT_RELU, "sigmoid": GEMV_ACT_SIGMOID, "silu": GEMV_ACT_SILU}

#: the C ABI's exported entry points (checked against include/gemv.h by the tests)
ENTRY_POINTS = ("gemv", "gemv_ex", "gemv_fused", "gemv_prepare", "gemv_plan", "gemv_last_config",
                "gemv_status_string", "gemv_last_cuda_error", "gemv_debug_inject",
                "gemv_release", "gemv_host", "gemv_splitk_noalloc",
                "gemv_wait_timeouts", "gemv_debug_wait_budget", "gla_decode", "gla_decode_ex")


class GemvConfig(ctypes.Structure):
    """Mirror of ``gemv_config`` in include/gemv.h."""
    _fields_ = [("variant", ctypes.c_int32), ("rows_per_warp", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32), ("warp_split", ctypes.c_int32),
                ("grid_split", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("k_segment", ctypes.c_int64), ("row_blocks", ctypes.c_int32),
                ("unroll", ctypes.c_int32), ("overlap", ctypes.c_int32),
                ("l2_prefetch", ctypes.c_int32), ("stages", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def to_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_ if f != "reserved"}


class GemvEpilogue(ctypes.Structure):
    """Mirror of ``gemv_epilogue`` in include/gemv.h."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("bias_dtype", ctypes.c_int32), ("activation", ctypes.c_int32)]


class GemvError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = gemv_status_string(status)
        if status == GEMV_ERR_CUDA:
            msg += f" (cudaError {gemv_last_cuda_error()})"
        super().__init__(f"{where}: status {status}: {msg}" if where else f"status {status}: {msg}")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"the GEMV CUDA library is not built ({path} missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` -- there is no fallback")
            L = ctypes.CDLL(path)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            cfgp = ctypes.POINTER(GemvConfig)
            L.gemv.argtypes = [vp, vp, vp, i64, i64, i32, vp]
            L.gemv_ex.argtypes = [vp, vp, vp, i64, i64, i32, cfgp, vp]
            L.gemv_fused.argtypes = [vp, i64, vp, vp, i64, i64, i32, ctypes.POINTER(GemvEpilogue), cfgp, vp]
            L.gemv_prepare.argtypes = [i64, i64, i32, i32, vp]
            L.gemv_plan.argtypes = [i64, i64, i32, i32, i32, cfgp, cfgp]
            L.gemv_last_config.argtypes = [cfgp]
            L.gemv_status_string.argtypes = [i32]
            L.gemv_status_string.restype = ctypes.c_char_p
            L.gemv_last_cuda_error.argtypes = []
            L.gemv_debug_inject.argtypes = [i32]
            L.gemv_release.argtypes = []
            L.gemv_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, vp]
            L.gemv_splitk_noalloc.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp]
            L.gemv_wait_timeouts.argtypes = [i32, ctypes.POINTER(ctypes.c_uint32)]
            L.gemv_debug_wait_budget.argtypes = [ctypes.c_int32]
            L.gla_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_float, i32, vp]
            L.gla_decode_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_float, i32, i32, i32, vp]
            for name in ENTRY_POINTS:
                if name != "gemv_status_string":
                    getattr(L, name).restype = i32
            _lib = L
    return _lib


# ------------------------------------------------------------- helpers --

def dtype_code(dtype: torch.dtype, out_fp32: bool = False) -> int:
    if dtype == torch.float16:
        return GEMV_F16_OUT_F32 if out_fp32 else GEMV_F16
    if dtype == torch.bfloat16:
        return GEMV_BF16_OUT_F32 if out_fp32 else GEMV_BF16
    raise TypeError(f"GEMV takes float16 or bfloat16 inputs, got {dtype}")


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _config_arg(config):
    if config is None:
        return None
    if isinstance(config, GemvConfig):
        return ctypes.byref(config)
    c = GemvConfig()
    for kname, v in dict(config).items():
        setattr(c, kname, int(v))
    return ctypes.byref(c)


def _check(status: int, where: str):
    if status != GEMV_OK:
        raise GemvError(status, where)


def _operands(B: torch.Tensor, a: torch.Tensor, c, out_fp32: bool):
    if B.dim() != 2 or a.dim() != 1 or B.shape[1] != a.shape[0]:
        raise ValueError(f"shape mismatch: B {tuple(B.shape)}, a {tuple(a.shape)}")
    if B.dtype != a.dtype:
        raise TypeError(f"B and a must share a dtype ({B.dtype} vs {a.dtype})")
    if not (B.is_cuda and a.is_cuda):
        raise ValueError("B and a must be CUDA tensors")
    n, k = B.shape
    if k > 0 and n > 0 and B.stride() != (k, 1):
        raise ValueError("B must be row-major with leading dimension k (contiguous rows)")
    if k > 1 and a.stride(0) != 1:
        raise ValueError("a must be contiguous")
    out_dtype = torch.float32 if out_fp32 else B.dtype
    if c is None:
        c = torch.empty(n, dtype=out_dtype, device=B.device)
    elif c.dtype != out_dtype or c.shape != (n,) or not c.is_cuda or (n > 1 and c.stride(0) != 1):
        raise ValueError(f"c must be a contiguous CUDA tensor of shape ({n},) and dtype {out_dtype}")
    if B.device != a.device or B.device != c.device:
        raise ValueError("B, a and c must be on the same device")
    return n, k, c


# ---------------------------------------------------------- entry points --

def gemv(B: torch.Tensor, a: torch.Tensor, c: torch.Tensor | None = None, out_fp32: bool = False,
         stream=None) -> torch.Tensor:
    """c = B @ a on B's device, asynchronously on ``stream`` (default: the
    current torch stream), launched as a programmatic dependent launch that
    reads and writes no memory before the preceding kernel has completed (it
    only asks L2 to prefetch its first tile of B).  Returns c (allocated if
    not given)."""
    n, k, c = _operands(B, a, c, out_fp32)
    with torch.cuda.device(B.device):
        st = lib().gemv(B.data_ptr(), a.data_ptr(), c.data_ptr(), n, k,
                        dtype_code(B.dtype, out_fp32), _stream_handle(stream))
    _check(st, "gemv")
    return c


def gemv_ex(B, a, c=None, out_fp32: bool = False, config=None, stream=None) -> torch.Tensor:
    """``gemv`` with a forced launch configuration (dict or GemvConfig;
    zero/missing fields are left to the planner, except ``overlap``, which
    is taken as given: 0 is a plain launch).  ``config=None`` is ``gemv``."""
    n, k, c = _operands(B, a, c, out_fp32)
    with torch.cuda.device(B.device):
        st = lib().gemv_ex(B.data_ptr(), a.data_ptr(), c.data_ptr(), n, k,
                           dtype_code(B.dtype, out_fp32), _config_arg(config), _stream_handle(stream))
    _check(st, "gemv_ex")
    return c


def gemv_fused(B, a, c=None, out_fp32: bool = False, alpha: float = 1.0, beta: float = 1.0, bias=None,
               activation: str = "none", config=None, stream=None) -> torch.Tensor:
    """c = act(alpha * (B @ a) + beta * bias), fused into the GEMV's store.
    ``B`` may be a row-strided view (stride (ldb, 1) with ldb >= k: rows of a
    larger matrix); ``bias`` (optional) is a CUDA tensor of n elements in B's
    dtype or float32; ``activation`` is 'none', 'relu', 'sigmoid' or 'silu'."""
    if B.dim() != 2 or a.dim() != 1 or B.shape[1] != a.shape[0]:
        raise ValueError(f"shape mismatch: B {tuple(B.shape)}, a {tuple(a.shape)}")
    n, k = B.shape
    if n > 0 and k > 0 and (B.stride(1) != 1 or B.stride(0) < k):
        raise ValueError("B must have unit column stride and row stride >= k")
    ldb = B.stride(0) if n > 1 else k
    out_dtype = torch.float32 if out_fp32 else B.dtype
    if c is None:
        c = torch.empty(n, dtype=out_dtype, device=B.device)
    if not (B.is_cuda and a.is_cuda and c.is_cuda) or c.dtype != out_dtype or c.shape != (n,):
        raise ValueError("B, a, c must be CUDA tensors; c of shape (n,) and the output dtype")
    if B.dtype != a.dtype or (k > 1 and a.stride(0) != 1) or (n > 1 and c.stride(0) != 1):
        raise ValueError("a must be contiguous with B's dtype; c contiguous")
    if B.device != a.device or B.device != c.device:
        raise ValueError("B, a and c must be on the same device")
    ep = GemvEpilogue()
    ep.alpha = float(alpha)
    ep.beta = float(beta)
    ep.activation = ACTIVATIONS[activation]
    if bias is not None:
        if not bias.is_cuda or bias.shape != (n,) or (n > 1 and bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous CUDA tensor of shape (n,)")
        if bias.dtype == torch.float32:
            ep.bias_dtype = GEMV_BIAS_F32
        elif bias.dtype == B.dtype:
            ep.bias_dtype = GEMV_BIAS_INPUT_TYPE
        else:
            raise TypeError("bias must be float32 or B's dtype")
        ep.bias = bias.data_ptr()
    with torch.cuda.device(B.device):
        st = lib().gemv_fused(B.data_ptr(), ldb, a.data_ptr(), c.data_ptr(), n, k,
                              dtype_code(B.dtype, out_fp32), ctypes.byref(ep), _config_arg(config),
                              _stream_handle(stream))
    _check(st, "gemv_fused")
    return c


def gemv_prepare(n: int, k: int, dtype: int, b_aligned16: bool = True, stream=None) -> None:
    _check(lib().gemv_prepare(n, k, dtype, 1 if b_aligned16 else 0, _stream_handle(stream)),
           "gemv_prepare")


def gemv_plan(n: int, k: int, dtype: int, b_aligned16: bool, sm_count: int, config=None) -> dict:
    """The planner's choice for a shape on a device with ``sm_count`` SMs
    (pure host function; needs no GPU)."""
    out = GemvConfig()
    _check(lib().gemv_plan(n, k, dtype, 1 if b_aligned16 else 0, sm_count, _config_arg(config),
                           ctypes.byref(out)), "gemv_plan")
    return out.to_dict()


def gemv_last_config() -> dict:
    out = GemvConfig()
    _check(lib().gemv_last_config(ctypes.byref(out)), "gemv_last_config")
    return out.to_dict()


def gemv_status_string(status: int) -> str:
    return lib().gemv_status_string(int(status)).decode()


def gemv_last_cuda_error() -> int:
    return int(lib().gemv_last_cuda_error())


def gemv_debug_inject(status: int) -> None:
    lib().gemv_debug_inject(int(status))


def gemv_release() -> None:
    lib().gemv_release()


def gemv_host(B_host: torch.Tensor, a_host: torch.Tensor, c_host: torch.Tensor, B_dev: torch.Tensor,
              a_dev: torch.Tensor, c_dev: torch.Tensor, stream=None) -> torch.Tensor:
    """End-to-end call from host buffers (pinned for true asynchrony): copies
    B and a into the device buffers, runs the GEMV, copies c back into
    ``c_host``.  Asynchronous on ``stream``; synchronize before reading c_host."""
    n, k = B_host.shape
    out_fp32 = c_host.dtype == torch.float32
    if B_host.is_cuda or a_host.is_cuda or c_host.is_cuda:
        raise ValueError("B_host, a_host and c_host must be host tensors")
    if not (B_host.is_contiguous() and a_host.is_contiguous() and c_host.is_contiguous()):
        raise ValueError("host buffers must be contiguous")
    _operands(B_dev, a_dev, c_dev, out_fp32)
    if B_dev.shape != B_host.shape or a_dev.shape != a_host.shape or c_dev.shape != c_host.shape:
        raise ValueError("host and device buffers must have the same shapes")
    with torch.cuda.device(B_dev.device):
        st = lib().gemv_host(B_host.data_ptr(), a_host.data_ptr(), c_host.data_ptr(), B_dev.data_ptr(),
                             a_dev.data_ptr(), c_dev.data_ptr(), n, k,
                             dtype_code(B_host.dtype, out_fp32), _stream_handle(stream))
    _check(st, "gemv_host")
    return c_host


def gemv_splitk_noalloc(B, a, c=None, out_fp32: bool = False, grid_split: int = 2, stream=None) -> torch.Tensor:
    """Split-K GEMV whose partial sums live in the library's fixed device
    scratch array instead of allocated memory (for callers that must not
    allocate while they run).  Calls that overlap on the GPU share that
    array and must not run concurrently."""
    n, k, c = _operands(B, a, c, out_fp32)
    with torch.cuda.device(B.device):
        st = lib().gemv_splitk_noalloc(B.data_ptr(), a.data_ptr(), c.data_ptr(), n, k,
                                       dtype_code(B.dtype, out_fp32), int(grid_split),
                                       _stream_handle(stream))
    _check(st, "gemv_splitk_noalloc")
    return c


def gemv_wait_timeouts(reset: bool = False) -> int:
    """Ring waits of the bulk variant that gave up on the current device
    (synchronizes the device); ``reset`` zeroes the counter after reading."""
    out = ctypes.c_uint32(0)
    _check(lib().gemv_wait_timeouts(1 if reset else 0, ctypes.byref(out)), "gemv_wait_timeouts")
    return int(out.value)


def gemv_debug_wait_budget(polls: int) -> None:
    """Test hook: the next bulk-variant launch polls each ring wait at most
    ``polls`` times (0: every wait gives up at once); -1 clears it."""
    _check(lib().gemv_debug_wait_budget(int(polls)), "gemv_debug_wait_budget")


def gla_decode(q, k, v, gk, S, scale: float, S_new=None, o=None, stream=None, variant: int = 0, flags: int = 0):
    """One gated-linear-attention decode step for bh heads: S_new =
    diag(exp(gk)) S + outer(k, v), o = scale * q^T S_new.  Shapes: q, k, gk
    (bh, dk); v (bh, dv); S (bh, dk, dv); one dtype (fp16, bf16 or fp32).
    ``S_new`` may be ``S`` (in place).  ``variant``: GLA_VARIANT_* (0: the
    library's choice); ``flags``: GLA_PREFETCH_STATE when no work in flight
    writes S (either calls ``gla_decode_ex``).  Returns (S_new, o)."""
    bh, dk, dv = S.shape
    if q.shape != (bh, dk) or k.shape != (bh, dk) or gk.shape != (bh, dk) or v.shape != (bh, dv):
        raise ValueError("shape mismatch")
    dt = S.dtype
    if dt not in _GLA_DTYPE or any(x.dtype != dt for x in (q, k, v, gk)):
        raise TypeError("q, k, v, gk, S must share one of float16, bfloat16, float32")
    if S_new is None:
        S_new = torch.empty_like(S)
    if o is None:
        o = torch.empty((bh, dv), dtype=dt, device=S.device)
    for x in (q, k, v, gk, S, S_new, o):
        if not x.is_cuda or not x.is_contiguous() or x.device != S.device:
            raise ValueError("all tensors must be contiguous CUDA tensors on one device")
    if S_new.shape != S.shape or S_new.dtype != dt or o.shape != (bh, dv) or o.dtype != dt:
        raise ValueError("S_new / o have the wrong shape or dtype")
    with torch.cuda.device(S.device):
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), gk.data_ptr(), S.data_ptr(), S_new.data_ptr(),
                o.data_ptr(), bh, dk, dv, float(scale), _GLA_DTYPE[dt])
        if variant or flags:
            st = lib().gla_decode_ex(*args, int(variant), int(flags), _stream_handle(stream))
        else:
            st = lib().gla_decode(*args, _stream_handle(stream))
    _check(st, "gla_decode")
    return S_new, o

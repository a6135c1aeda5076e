"""Oracle for the GEMV ``c = B @ a`` -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product path (the CUDA library
``memory_bound_gemv_02_gb300`` and its C-ABI) never imports it, and this
package imports nothing from there.

The arithmetic lives in ``gemv_ref.c`` (plain C, binary64, one thread, one row
at a time, ascending column index), a direct restatement of the definition in
TileLang Case Studies, Case B "Background": B is (n, k) row-major, a is (k,),
``c_i = sum_j B[i, j] a[j]``.  This module only loads the compiled library
(building it with gcc when it is missing or older than its source) and
marshals numpy arrays.

Every function is pinned by ``tests/test_oracle.py`` against things other than
itself: torch/numpy casts for the decoders and encoders, closed forms (ones,
identity), exact rational sums, numpy's float64 matmul and integer-input
invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemv_ref.c")
_LIB = os.path.join(_HERE, "libgemv_ref.so")

#: format codes of gemv_ref.c
FMT = {"f16": 0, "bf16": 1, "f32": 2}
#: activation codes of gemv_ref.c
ACT = {"none": 0, "relu": 1, "sigmoid": 2, "silu": 3}

_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``gemv_ref.c`` into ``libgemv_ref.so`` next to it (gcc, -O2,
    no fast-math, no FMA contraction).  Returns the library path."""
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _ptr(arr: np.ndarray) -> int:
    return arr.ctypes.data


def _bits16(x) -> np.ndarray:
    arr = np.ascontiguousarray(x)
    if arr.dtype != np.uint16:
        raise TypeError(f"expected uint16 bit patterns, got {arr.dtype}")
    return arr


class Oracle:
    """The oracle's entry points bound to one compiled copy of ``gemv_ref.c``."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.gemv_ref_decode_array.argtypes = [vp, i64, ctypes.c_int, vp]
        lib.gemv_ref_decode_array.restype = None
        lib.gemv_ref_encode_array.argtypes = [vp, i64, ctypes.c_int, vp]
        lib.gemv_ref_encode_array.restype = None
        lib.gemv_ref.argtypes = [vp, vp, i64, i64, ctypes.c_int, vp, vp]
        lib.gemv_ref.restype = ctypes.c_int
        lib.gemv_ref_rows.argtypes = [vp, vp, i64, i64, ctypes.c_int, vp, i64, vp, vp]
        lib.gemv_ref_rows.restype = ctypes.c_int
        lib.gemv_ref_epilogue.argtypes = [vp, vp, i64, ctypes.c_double, ctypes.c_double, vp, ctypes.c_int,
                                          ctypes.c_int, vp, vp]
        lib.gemv_ref_epilogue.restype = ctypes.c_int
        lib.gla_ref_decode.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_double, ctypes.c_int,
                                       vp, vp, vp, vp]
        lib.gla_ref_decode.restype = ctypes.c_int
        self.lib = lib

    def decode(self, bits, fmt: str) -> np.ndarray:
        """Decode uint16 bit patterns of ``fmt`` ('f16' or 'bf16') to float64."""
        b = _bits16(bits)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.gemv_ref_decode_array(_ptr(b), b.size, FMT[fmt], _ptr(out))
        return out

    def encode(self, x, fmt: str) -> np.ndarray:
        """Round float64 values to ``fmt`` ('f16', 'bf16' or 'f32'), nearest-even.
        Returns uint16 patterns for the 16-bit formats, uint32 for 'f32'."""
        v = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(v.shape, dtype=np.uint32 if fmt == "f32" else np.uint16)
        self.lib.gemv_ref_encode_array(_ptr(v), v.size, FMT[fmt], _ptr(out))
        return out

    def gemv_ref(self, B_bits, a_bits, fmt: str):
        """Oracle GEMV.  ``B_bits`` (n, k) and ``a_bits`` (k,) are uint16 bit
        patterns of ``fmt`` ('f16' or 'bf16').  Returns float64 arrays
        ``(c, s)`` with ``c_i = sum_j B_ij a_j`` and ``s_i = sum_j |B_ij a_j|``."""
        B = _bits16(B_bits)
        a = _bits16(a_bits)
        if B.ndim != 2 or a.ndim != 1 or B.shape[1] != a.shape[0]:
            raise ValueError(f"shape mismatch: B {B.shape}, a {a.shape}")
        n, k = B.shape
        c = np.zeros(n, dtype=np.float64)
        s = np.zeros(n, dtype=np.float64)
        rc = self.lib.gemv_ref(_ptr(B), _ptr(a), n, k, FMT[fmt], _ptr(c), _ptr(s))
        if rc != 0:
            raise ValueError("gemv_ref rejected its arguments")
        return c, s

    def gemv_ref_rows(self, B_bits, a_bits, fmt: str, rows):
        """Oracle results for the listed rows of ``B_bits`` only."""
        B = _bits16(B_bits)
        a = _bits16(a_bits)
        n, k = B.shape
        r = np.ascontiguousarray(rows, dtype=np.int64)
        c = np.zeros(r.size, dtype=np.float64)
        s = np.zeros(r.size, dtype=np.float64)
        rc = self.lib.gemv_ref_rows(_ptr(B), _ptr(a), n, k, FMT[fmt], _ptr(r), r.size, _ptr(c),
                                    _ptr(s))
        if rc != 0:
            raise ValueError("gemv_ref_rows rejected its arguments")
        return c, s

    def round_out(self, c, out_fmt: str) -> np.ndarray:
        """Round oracle results to the output format's bit patterns."""
        return self.encode(c, out_fmt)

    def gemv_ref_epilogue(self, c, s, alpha=1.0, beta=0.0, bias_bits=None, bias_fmt="f32",
                          act: str = "none"):
        """y = act(alpha * c + beta * bias) in binary64 and the tolerance scale
        (|alpha| s + |beta bias|) * max slope of act.  ``bias_bits``: uint16
        patterns of 'f16'/'bf16' or uint32 patterns of 'f32', or None."""
        c = np.ascontiguousarray(c, dtype=np.float64)
        s = np.ascontiguousarray(s, dtype=np.float64)
        n = c.size
        y = np.zeros(n, dtype=np.float64)
        scale = np.zeros(n, dtype=np.float64)
        bptr = None
        if bias_bits is not None:
            bias_bits = np.ascontiguousarray(bias_bits)
            want = np.uint32 if bias_fmt == "f32" else np.uint16
            if bias_bits.dtype != want or bias_bits.size != n:
                raise TypeError("bias bit patterns of the wrong type or size")
            bptr = _ptr(bias_bits)
        rc = self.lib.gemv_ref_epilogue(_ptr(c), _ptr(s), n, float(alpha), float(beta), bptr, FMT[bias_fmt],
                                        ACT[act], _ptr(y), _ptr(scale))
        if rc != 0:
            raise ValueError("gemv_ref_epilogue rejected its arguments")
        return y, scale


    def gla_ref_decode(self, q, k, v, gk, S, scale: float, fmt: str):
        """One GLA decode step for bh heads.  Bit-pattern arrays of ``fmt``
        ('f16'/'bf16': uint16, 'f32': uint32): q, k, gk (bh, dk), v (bh, dv),
        S (bh, dk, dv).  Returns binary64 (S_new, o, S_scale, o_scale)."""
        want = np.uint32 if fmt == "f32" else np.uint16
        arrs = [np.ascontiguousarray(x) for x in (q, k, v, gk, S)]
        if any(x.dtype != want for x in arrs):
            raise TypeError(f"expected {want.__name__} bit patterns for {fmt}")
        q, k, v, gk, S = arrs
        bh, dk, dv = S.shape
        if q.shape != (bh, dk) or k.shape != (bh, dk) or gk.shape != (bh, dk) or v.shape != (bh, dv):
            raise ValueError("shape mismatch")
        S_new = np.zeros((bh, dk, dv))
        ss = np.zeros((bh, dk, dv))
        o = np.zeros((bh, dv))
        os_ = np.zeros((bh, dv))
        rc = self.lib.gla_ref_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(gk), _ptr(S), bh, dk, dv, float(scale),
                                     FMT[fmt], _ptr(S_new), _ptr(o), _ptr(ss), _ptr(os_))
        if rc != 0:
            raise ValueError("gla_ref_decode rejected its arguments")
        return S_new, o, ss, os_


def default() -> Oracle:
    """The oracle built from this directory's ``gemv_ref.c``."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def decode(bits, fmt):
    return default().decode(bits, fmt)


def encode(x, fmt):
    return default().encode(x, fmt)


def gemv_ref(B_bits, a_bits, fmt):
    return default().gemv_ref(B_bits, a_bits, fmt)


def gemv_ref_rows(B_bits, a_bits, fmt, rows):
    return default().gemv_ref_rows(B_bits, a_bits, fmt, rows)


def round_out(c, out_fmt):
    return default().round_out(c, out_fmt)


def gemv_ref_epilogue(c, s, alpha=1.0, beta=0.0, bias_bits=None, bias_fmt="f32", act="none"):
    return default().gemv_ref_epilogue(c, s, alpha, beta, bias_bits, bias_fmt, act)


def gla_ref_decode(q, k, v, gk, S, scale, fmt):
    return default().gla_ref_decode(q, k, v, gk, S, scale, fmt)

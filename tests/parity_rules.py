"""Acceptance rules for comparing a GEMV result with the oracle.

* 16-bit output (fp16/bf16): |c - c_ref| <= 1e-2 * max(1, |c_ref|), with c_ref
  the oracle's unrounded binary64 value.
* fp32 output: |c - c_ref| <= 1e-5 * S, S = sum_j |B_ij a_j|.
* Hard failure, whatever the tolerance: an error larger than one unit in the
  last place of the output format that is exactly a power of two 2^m with
  m >= -4 (0.0625, 0.125, 0.25, ...).  TileLang Case Studies, Case A
  ("Symptoms", "Lessons") identifies such round errors as the fingerprint of
  a systematic design bug rather than of rounding.
* Non-finite oracle values must be matched in kind (same inf, or NaN).
"""
from __future__ import annotations

import numpy as np

FMT_PARAMS = {"f16": (10, -14), "bf16": (7, -126), "f32": (23, -126)}


def ulp(x, fmt: str) -> np.ndarray:
    """Spacing of ``fmt`` values at |x| (the quantum of x's binade)."""
    mbits, emin = FMT_PARAMS[fmt]
    ax = np.abs(np.asarray(x, dtype=np.float64))
    ok = np.isfinite(ax) & (ax > 0)
    _, e = np.frexp(np.where(ok, ax, 1.0))
    E = np.maximum(np.where(ok, e - 1, emin), emin)
    return np.ldexp(1.0, E - mbits)


def pow2_errors(err, c_ref, fmt: str) -> np.ndarray:
    """Mask of errors that are exact powers of two >= 2^-4 and above 1 ulp."""
    e = np.abs(np.asarray(err, dtype=np.float64))
    mant, _ = np.frexp(np.where(np.isfinite(e) & (e > 0), e, 3.0))
    is_pow2 = (mant == 0.5) & np.isfinite(e) & (e > 0)
    return is_pow2 & (e >= 2.0 ** -4) & (e > ulp(c_ref, fmt))


def check(c_gpu, c_ref, s_ref, out_fmt: str, label: str = "") -> dict:
    """Assert that ``c_gpu`` (float64 values of the output) passes; return stats."""
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    c_ref = np.asarray(c_ref, dtype=np.float64)
    s_ref = np.asarray(s_ref, dtype=np.float64)
    assert c_gpu.shape == c_ref.shape, (label, c_gpu.shape, c_ref.shape)
    fin = np.isfinite(c_ref)
    # non-finite reference entries: same infinity, or NaN for NaN
    nf = ~fin
    if nf.any():
        same = (np.isnan(c_ref[nf]) & np.isnan(c_gpu[nf])) | (c_ref[nf] == c_gpu[nf])
        assert same.all(), f"{label}: non-finite mismatch at rows {np.flatnonzero(nf)[~same][:8]}"
    if out_fmt == "f32":
        tol = 1e-5 * s_ref
    else:
        tol = 1e-2 * np.maximum(1.0, np.abs(c_ref))
    err = np.where(fin, c_gpu - c_ref, 0.0)
    p2 = fin & pow2_errors(err, c_ref, out_fmt)
    if p2.any():
        i = np.flatnonzero(p2)[:8]
        raise AssertionError(f"{label}: power-of-two error pattern at rows {i.tolist()}: "
                             f"{err[i].tolist()}")
    bad = fin & ~(np.abs(err) <= tol)
    if bad.any():
        i = np.flatnonzero(bad)[:8]
        raise AssertionError(f"{label}: {bad.sum()} rows out of tolerance; rows {i.tolist()} "
                             f"gpu {c_gpu[i].tolist()} ref {c_ref[i].tolist()} tol {tol[i].tolist()}")
    aerr = np.abs(err)
    j = int(np.argmax(aerr)) if aerr.size else 0
    return {"max_err": float(aerr.max()) if aerr.size else 0.0, "argmax": j,
            "max_rel_tol": float((aerr / np.maximum(tol, 1e-300)).max()) if aerr.size else 0.0}

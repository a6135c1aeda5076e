"""Shared helpers of the GPU tests: run the CUDA path through the C-ABI
binding and compare with the oracle on the same bits."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import parity_rules
from memory_bound_gemv_02_gb300 import inputs


def fmt_of(t: torch.Tensor) -> str:
    return "f16" if t.dtype == torch.float16 else "bf16"


def sample_rows(n: int, m: int = 192, seed: int = 0) -> np.ndarray:
    """First and last rows plus a seeded random sample in between."""
    if n <= m:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    edge = min(32, n // 4)
    mid = rng.choice(np.arange(edge, n - edge), size=m - 2 * edge, replace=False)
    return np.unique(np.concatenate([np.arange(edge), np.arange(n - edge, n), mid]))


def oracle_chunked(B_bits: np.ndarray, a_bits: np.ndarray, fmt: str, chunk_rows: int = 2048):
    """The oracle over every row of ``B_bits``, row chunks run on a pool of
    host threads (each chunk is one unchanged oracle call; rows are
    independent, so the result equals one call over the whole matrix)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    n = B_bits.shape[0]
    c = np.empty(n, dtype=np.float64)
    s = np.empty(n, dtype=np.float64)

    def one(i0):
        ci, si = oracle.gemv_ref(B_bits[i0:i0 + chunk_rows], a_bits, fmt)
        c[i0:i0 + chunk_rows] = ci
        s[i0:i0 + chunk_rows] = si

    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(one, range(0, n, chunk_rows)))
    return c, s


def oracle_for(B: torch.Tensor, a: torch.Tensor, rows=None):
    fmt = fmt_of(B)
    a_bits = inputs.to_bits(a)
    if rows is None:
        if B.numel() >= (1 << 26):  # large: rows in parallel chunks
            return oracle_chunked(inputs.to_bits(B), a_bits, fmt)
        return oracle.gemv_ref(inputs.to_bits(B), a_bits, fmt)
    idx = torch.as_tensor(np.asarray(rows), device=B.device, dtype=torch.long)
    return oracle.gemv_ref(inputs.to_bits(B.index_select(0, idx)), a_bits, fmt)


def gpu_values(c: torch.Tensor, rows=None) -> np.ndarray:
    if rows is not None:
        c = c.index_select(0, torch.as_tensor(np.asarray(rows), device=c.device, dtype=torch.long))
    return c.double().cpu().numpy()


def check_against_oracle(c: torch.Tensor, B: torch.Tensor, a: torch.Tensor, out_fp32: bool, rows=None,
                         label: str = "") -> dict:
    torch.cuda.synchronize()
    c_ref, s_ref = oracle_for(B, a, rows)
    out_fmt = "f32" if out_fp32 else fmt_of(B)
    return parity_rules.check(gpu_values(c, rows), c_ref, s_ref, out_fmt, label)


def exact_bits_match(c: torch.Tensor, B: torch.Tensor, a: torch.Tensor, out_fp32: bool) -> bool:
    """Integer-valued inputs: the output must equal the oracle rounded once."""
    torch.cuda.synchronize()
    c_ref, _ = oracle_for(B, a)
    out_fmt = "f32" if out_fp32 else fmt_of(B)
    want = oracle.round_out(c_ref, out_fmt)
    got = inputs.out_bits(c)
    return bool((got == want).all())

"""Seeded synthetic inputs for the GEMV ``c = B @ a``.

This module draws random numbers and moves bit patterns around; it holds none
of the product's arithmetic.  Both the CUDA path's callers (tests, benchmark)
and the oracle's callers use it, so that both sides see the same bits.

Recipe (the shapes and distributions of the workloads in TileLang Case
Studies, Cases B-B.3, made synthetic): one ``torch.Generator`` on the target
device seeded with ``seed``; B (n, k) is drawn first, then a (k,);
``uniform`` is ``2 * rand - 1`` (uniform on [-1, 1)), ``normal`` is
``randn * sigma``; both are drawn in float32 and cast (round to nearest even)
to float16 or bfloat16.
"""
from __future__ import annotations

import numpy as np
import torch

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def make_inputs(n: int, k: int, dtype: str, dist: str = "uniform", seed: int = 0,
                device="cpu", b_sigma: float = 0.02, a_sigma: float = 1.0):
    """Return ``(B, a)`` torch tensors of ``dtype`` ('f16'/'bf16') on ``device``.

    ``dist='uniform'``: B and a uniform on [-1, 1).  ``dist='normal'``: B
    normal(0, b_sigma), a normal(0, a_sigma)."""
    g = generator(seed, device)
    td = TORCH_DTYPE[dtype]
    if dist == "uniform":
        B = (torch.rand((n, k), generator=g, device=device, dtype=torch.float32) * 2 - 1).to(td)
        a = (torch.rand((k,), generator=g, device=device, dtype=torch.float32) * 2 - 1).to(td)
    elif dist == "normal":
        B = (torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * b_sigma).to(td)
        a = (torch.randn((k,), generator=g, device=device, dtype=torch.float32) * a_sigma).to(td)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return B, a


def make_int_inputs(n: int, k: int, dtype: str, seed: int = 0, device="cpu", lo: int = -3,
                    hi: int = 3):
    """Integer-valued B and a, uniform on {lo..hi}: every partial sum of a
    row is an integer far below 2^24, so it is exact in float32 in any
    summation order."""
    g = generator(seed, device)
    td = TORCH_DTYPE[dtype]
    B = torch.randint(lo, hi + 1, (n, k), generator=g, device=device, dtype=torch.int32).to(td)
    a = torch.randint(lo, hi + 1, (k,), generator=g, device=device, dtype=torch.int32).to(td)
    return B, a


def to_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a float16/bfloat16 tensor's bit patterns as uint16."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(bits: np.ndarray, dtype: str, device="cpu") -> torch.Tensor:
    """Tensor of ``dtype`` whose elements carry the given uint16 patterns."""
    arr = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(arr.view(np.int16).copy()).view(TORCH_DTYPE[dtype]).to(device)


def out_bits(c: torch.Tensor) -> np.ndarray:
    """Host bit patterns of an output tensor: uint16 for 16-bit, uint32 for float32."""
    c = c.detach().contiguous().cpu()
    if c.dtype == torch.float32:
        return c.view(torch.int32).numpy().view(np.uint32)
    return c.view(torch.int16).numpy().view(np.uint16)

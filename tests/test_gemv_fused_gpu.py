"""The fused epilogue and row-strided B (gemv_fused), against the oracle.

c[i] = act(alpha * sum_{j<k} B[i*ldb + j] a[j] + beta * bias[i]) with act in
{none, relu, sigmoid, silu}, bias in the input type or fp32 (the register
epilogue of the TileLang optimization guide, "Epilogue Fusion").  The oracle
applies the same epilogue in binary64 to its binary64 sums.

Tolerances: 16-bit output 1e-2 * max(1, |y_ref|); fp32 output
1e-5 * (|alpha| S + |beta bias|) * max slope(act) + 2e-6 |y_ref| (the
epilogue's own fp32 rounding and exp); plus the power-of-two rule.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import memory_bound_gemv_02_gb300 as g
import oracle
import parity_rules
from gpu_helpers import fmt_of, gpu_values
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu


def _reference(B, a, alpha, beta, bias, act):
    fmt = fmt_of(B)
    c, s = oracle.gemv_ref(inputs.to_bits(B.contiguous()), inputs.to_bits(a), fmt)
    if bias is None:
        return oracle.gemv_ref_epilogue(c, s, alpha, beta, None, "f32", act)
    if bias.dtype == torch.float32:
        bits = bias.cpu().numpy().view(np.uint32)
        return oracle.gemv_ref_epilogue(c, s, alpha, beta, bits, "f32", act)
    return oracle.gemv_ref_epilogue(c, s, alpha, beta, inputs.to_bits(bias), fmt, act)


def _check(y, B, a, alpha, beta, bias, act, out_fp32, label):
    torch.cuda.synchronize()
    y_ref, scale = _reference(B, a, alpha, beta, bias, act)
    got = gpu_values(y)
    out_fmt = "f32" if out_fp32 else fmt_of(B)
    if out_fp32:
        tol = 1e-5 * scale + 2e-6 * np.abs(y_ref) + 1e-30
    else:
        tol = 1e-2 * np.maximum(1.0, np.abs(y_ref))
    err = got - y_ref
    p2 = parity_rules.pow2_errors(err, y_ref, out_fmt)
    assert not p2.any(), f"{label}: power-of-two errors at {np.flatnonzero(p2)[:5]}"
    bad = ~(np.abs(err) <= tol)
    assert not bad.any(), (f"{label}: {int(bad.sum())} rows off; first {np.flatnonzero(bad)[:5]} "
                           f"got {got[bad][:3]} ref {y_ref[bad][:3]}")


ACTS = ["none", "relu", "sigmoid", "silu"]


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bias_kind", [None, "input", "f32"])
@pytest.mark.parametrize("out_fp32", [False, True])
def test_epilogue_parity(cuda_dev, act, dtype, bias_kind, out_fp32):
    n, k = 1031, 4099
    B, a = inputs.make_inputs(n, k, dtype, "uniform", 3, cuda_dev)
    B = B * 0.05
    bias = None
    if bias_kind is not None:
        bdt = torch.float32 if bias_kind == "f32" else B.dtype
        bias = (torch.rand(n, generator=inputs.generator(9, cuda_dev), device=cuda_dev) * 4 - 2).to(bdt)
    for cfg in (None, {"grid_split": 3}, {"variant": 2}, {"warp_split": 4, "overlap": 2}):
        y = g.gemv_fused(B, a, out_fp32=out_fp32, alpha=1.5, beta=-0.75, bias=bias, activation=act, config=cfg)
        _check(y, B, a, 1.5, -0.75, bias, act, out_fp32, f"{act} {dtype} bias={bias_kind} {cfg}")


@pytest.mark.parametrize("n,k,pad", [(300, 1000, 8), (300, 1000, 3), (129, 4096, 64), (129, 4096, 1),
                                     (77, 7169, 7), (513, 64, 0), (2000, 512, 24)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_strided_rows(cuda_dev, n, k, pad, dtype):
    """B is the first k columns of an (n, k + pad) buffer whose padding holds
    NaN: the padding must never reach a row's result."""
    ldb = k + pad
    buf = torch.full((n, ldb), float("nan"), dtype=inputs.TORCH_DTYPE[dtype], device=cuda_dev)
    Bc, a = inputs.make_inputs(n, k, dtype, "uniform", 4, cuda_dev)
    buf[:, :k] = Bc
    Bv = buf[:, :k]
    assert Bv.stride() == (ldb, 1)
    for cfg in (None, {"grid_split": 2}, {"warp_split": 2}, {"overlap": 3}):
        for out_fp32 in (False, True):
            y = g.gemv_fused(Bv, a, out_fp32=out_fp32, config=cfg)
            _check(y, Bc, a, 1.0, 0.0, None, "none", out_fp32, f"ldb={ldb} {cfg} f32={out_fp32}")
    if k % 8 == 0 and ldb % 8 == 0:
        g.gemv_fused(Bv, a)
        assert g.gemv_last_config()["variant"] == g.GEMV_VARIANT_TILES


def test_identity_epilogue_is_gemv_bitwise(cuda_dev):
    B, a = inputs.make_inputs(3001, 5000, "bf16", "normal", 1, cuda_dev)
    for out_fp32 in (False, True):
        ref = g.gemv(B, a, out_fp32=out_fp32)
        got = g.gemv_fused(B, a, out_fp32=out_fp32, alpha=1.0, beta=0.0)
        torch.cuda.synchronize()
        assert (inputs.out_bits(got) == inputs.out_bits(ref)).all()


def test_empty_k_with_epilogue(cuda_dev):
    n = 70
    B = torch.empty((n, 0), dtype=torch.float16, device=cuda_dev)
    a = torch.empty(0, dtype=torch.float16, device=cuda_dev)
    bias = torch.linspace(-3, 3, n, device=cuda_dev)
    y = g.gemv_fused(B, a, out_fp32=True, beta=2.0, bias=bias, activation="sigmoid")
    torch.cuda.synchronize()
    zeros = np.zeros(n)
    want, _ = oracle.gemv_ref_epilogue(zeros, zeros, 1.0, 2.0, bias.cpu().numpy().view(np.uint32), "f32",
                                       "sigmoid")
    assert (np.abs(y.double().cpu().numpy() - want) <= 2e-6 * np.abs(want)).all()


def test_fused_argument_errors(cuda_dev):
    B, a = inputs.make_inputs(64, 128, "f16", "uniform", 0, cuda_dev)
    with pytest.raises(KeyError):
        g.gemv_fused(B, a, activation="tanh")
    with pytest.raises(TypeError):
        g.gemv_fused(B, a, bias=torch.zeros(64, dtype=torch.bfloat16, device=cuda_dev))

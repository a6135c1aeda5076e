"""Pins for the oracle's GLA decode step (CPU only).

One step of gated linear attention (TileLang Case Studies, Case D
"Background"): S_new = diag(exp(gk)) S + outer(k, v), o = scale * q^T S_new,
per head.  The pins use what the definition fixes exactly: exp(0) = 1 and
exp(-inf) = 0 give closed forms; small integer inputs make every sum exact;
heads are independent; the row/column layout is checked by unit vectors.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from memory_bound_gemv_02_gb300 import inputs


def _bits(x, fmt):
    x = np.asarray(x, dtype=np.float64)
    if fmt == "f32":
        return x.astype(np.float32).view(np.uint32)
    return inputs.to_bits(torch.from_numpy(x.astype(np.float32)).to(inputs.TORCH_DTYPE[fmt]))


def _decode(bits, fmt):
    if fmt == "f32":
        return bits.view(np.float32).astype(np.float64)
    return inputs.from_bits(bits, fmt).double().numpy()


def _int_case(bh, dk, dv, seed, lo=-3, hi=3):
    rng = np.random.default_rng(seed)
    q = rng.integers(lo, hi + 1, (bh, dk)).astype(np.float64)
    k = rng.integers(lo, hi + 1, (bh, dk)).astype(np.float64)
    v = rng.integers(lo, hi + 1, (bh, dv)).astype(np.float64)
    S = rng.integers(lo, hi + 1, (bh, dk, dv)).astype(np.float64)
    return q, k, v, S


@pytest.mark.parametrize("fmt", ["f16", "bf16", "f32"])
def test_no_decay_integer_inputs_exact(fmt):
    """gk = 0: S_new = S + k v^T and o = scale q^T S_new, all exact."""
    bh, dk, dv = 3, 5, 7
    q, k, v, S = _int_case(bh, dk, dv, 1)
    gk = np.zeros((bh, dk))
    S_new, o, ss, os_ = oracle.gla_ref_decode(_bits(q, fmt), _bits(k, fmt), _bits(v, fmt), _bits(gk, fmt),
                                              _bits(S, fmt), 0.5, fmt)
    for h in range(bh):
        for i in range(dk):
            for j in range(dv):
                assert S_new[h, i, j] == S[h, i, j] + k[h, i] * v[h, j]
                assert ss[h, i, j] == abs(S[h, i, j]) + abs(k[h, i] * v[h, j])
        for j in range(dv):
            exact = sum(int(q[h, i]) * int(S[h, i, j] + k[h, i] * v[h, j]) for i in range(dk))
            assert o[h, j] == 0.5 * exact
            assert os_[h, j] == 0.5 * sum(abs(int(q[h, i]) * int(S[h, i, j] + k[h, i] * v[h, j]))
                                          for i in range(dk))


@pytest.mark.parametrize("fmt", ["f16", "bf16", "f32"])
def test_full_decay_forgets_state(fmt):
    """gk = -inf: exp = 0, so S_new = k v^T whatever S held."""
    bh, dk, dv = 2, 4, 8
    q, k, v, S = _int_case(bh, dk, dv, 2)
    S = S * 1000.0
    gk = np.full((bh, dk), -np.inf)
    S_new, o, _, _ = oracle.gla_ref_decode(_bits(q, fmt), _bits(k, fmt), _bits(v, fmt), _bits(gk, fmt),
                                           _bits(S, fmt), 1.0, fmt)
    expect = k[:, :, None] * v[:, None, :]
    assert (S_new == expect).all()
    assert (o == np.einsum("hi,hij->hj", q, expect)).all()


def test_unit_query_reads_one_state_row():
    """q = e_r picks row r of S_new: pins the row/column layout and scale."""
    bh, dk, dv = 2, 6, 4
    q, k, v, S = _int_case(bh, dk, dv, 3)
    gk = np.zeros((bh, dk))
    for r in range(dk):
        qe = np.zeros((bh, dk))
        qe[:, r] = 1.0
        S_new, o, _, _ = oracle.gla_ref_decode(_bits(qe, "f32"), _bits(k, "f32"), _bits(v, "f32"),
                                               _bits(gk, "f32"), _bits(S, "f32"), -2.0, "f32")
        assert (o == -2.0 * S_new[:, r, :]).all()


def test_heads_are_independent():
    bh, dk, dv = 4, 3, 5
    q, k, v, S = _int_case(bh, dk, dv, 4)
    gk = np.random.default_rng(5).uniform(-2, 0, (bh, dk))
    args = [_bits(x, "bf16") for x in (q, k, v, gk, S)]
    S_new, o, _, _ = oracle.gla_ref_decode(*args, 0.25, "bf16")
    perm = np.array([2, 0, 3, 1])
    S_p, o_p, _, _ = oracle.gla_ref_decode(*[np.ascontiguousarray(a[perm]) for a in args], 0.25, "bf16")
    assert (S_p == S_new[perm]).all() and (o_p == o[perm]).all()


def test_exact_rationals_with_unit_decay():
    """A 1x3x2 head with dyadic values, against Fraction arithmetic."""
    q = np.array([[0.5, -1.25, 2.0]])
    k = np.array([[1.5, 0.25, -0.75]])
    v = np.array([[3.0, -0.5]])
    S = np.array([[[1.0, 2.0], [-4.0, 0.125], [0.375, -8.0]]])
    gk = np.zeros((1, 3))
    S_new, o, _, _ = oracle.gla_ref_decode(*[_bits(x, "f16") for x in (q, k, v, gk, S)], 0.125, "f16")
    for j in range(2):
        sn = [Fraction(S[0, i, j]) + Fraction(k[0, i]) * Fraction(v[0, j]) for i in range(3)]
        for i in range(3):
            assert Fraction(S_new[0, i, j]) == sn[i]
        assert Fraction(o[0, j]) == Fraction(1, 8) * sum(Fraction(q[0, i]) * sn[i] for i in range(3))


@pytest.mark.parametrize("fmt", ["f16", "bf16", "f32"])
def test_numpy_cross_check(fmt):
    """numpy float64 (exp, outer, matmul) on the decoded inputs agrees within
    the binary64 error bound."""
    rng = np.random.default_rng(6)
    bh, dk, dv = 5, 16, 24
    vals = [rng.uniform(-1, 1, (bh, dk)), rng.uniform(-1, 1, (bh, dk)), rng.uniform(-1, 1, (bh, dv)),
            rng.uniform(-3, 0.5, (bh, dk)), rng.uniform(-2, 2, (bh, dk, dv))]
    bits = [_bits(x, fmt) for x in vals]
    q, k, v, gk, S = [_decode(b, fmt) for b in bits]
    S_new, o, ss, os_ = oracle.gla_ref_decode(*bits, 0.125, fmt)
    ref_S = np.exp(gk)[:, :, None] * S + k[:, :, None] * v[:, None, :]
    ref_o = 0.125 * np.einsum("hi,hij->hj", q, ref_S)
    assert (np.abs(S_new - ref_S) <= 4 * 2.0 ** -53 * ss).all()
    assert (np.abs(o - ref_o) <= 2 * dk * 2.0 ** -53 * (os_ + np.abs(ref_o)) + 1e-300).all()


def test_f32_decode_matches_numpy():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32)
    with np.errstate(invalid="ignore"):  # NaN patterns among the random bits
        vals = bits.view(np.float32).astype(np.float64)
    fin = np.isfinite(vals)
    one = np.zeros((1, 1), np.uint32)
    for b, want in zip(bits[fin][:2000], vals[fin][:2000]):
        S_new, _, _, _ = oracle.gla_ref_decode(one, one, one.reshape(1, 1), one,
                                               np.array([[[b]]], np.uint32), 1.0, "f32")
        assert S_new[0, 0, 0] == want  # exp(0) * S + 0 * 0


def test_bad_arguments():
    z = np.zeros((1, 2), np.uint16)
    with pytest.raises(TypeError):
        oracle.gla_ref_decode(z, z, z, z, np.zeros((1, 2, 2), np.uint32), 1.0, "f16")
    with pytest.raises(ValueError):
        oracle.gla_ref_decode(z, z, np.zeros((1, 3), np.uint16), z, np.zeros((1, 2, 2), np.uint16), 1.0, "f16")
    assert math.isclose(math.exp(0.0), 1.0)

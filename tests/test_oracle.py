"""Pins for the oracle (CPU only).

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (a dropped term, a wrong sign, a transposed operand, a
wrong row stride, a bad exponent bias, double rounding) fails at least one.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import parity_rules
from memory_bound_gemv_02_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- decoding --

@pytest.mark.parametrize("fmt,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_decode_exhaustive(fmt, tdt):
    """All 2^16 patterns decode exactly as torch's CPU widening does."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, fmt)
    theirs = torch.from_numpy(bits.view(np.int16).copy()).view(tdt).double().numpy()
    nan_o, nan_t = np.isnan(ours), np.isnan(theirs)
    assert (nan_o == nan_t).all()
    assert (ours[~nan_o] == theirs[~nan_t]).all()
    # signed zeros survive
    assert np.signbit(ours[~nan_o]).tolist() == np.signbit(theirs[~nan_t]).tolist()


def test_decode_f16_against_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, "f16")
    theirs = bits.view(np.float16).astype(np.float64)
    m = ~np.isnan(theirs)
    assert (ours[m] == theirs[m]).all() and np.isnan(ours[~m]).all()


def test_decode_known_values():
    # format definitions: fp16 1.0 = 0x3C00, 65504 = 0x7BFF, min subnormal 0x0001 = 2^-24;
    # bf16 1.0 = 0x3F80, -2.0 = 0xC000, min subnormal 0x0001 = 2^-133
    assert oracle.decode(np.array([0x3C00, 0x7BFF, 0x0001, 0x8400], np.uint16), "f16").tolist() == \
        [1.0, 65504.0, 2.0 ** -24, -(2.0 ** -14)]
    assert oracle.decode(np.array([0x3F80, 0xC000, 0x0001, 0x7F7F], np.uint16), "bf16").tolist() == \
        [1.0, -2.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127]


# ---------------------------------------------------------------- encoding --

def _log_uniform(rng, count, lo, hi):
    mag = np.exp2(rng.uniform(lo, hi, count))
    return np.where(rng.random(count) < 0.5, -mag, mag)


def test_encode_f16_against_numpy():
    """numpy converts binary64 to binary16 directly with nearest-even."""
    rng = np.random.default_rng(1)
    x = np.concatenate([_log_uniform(rng, 400_000, -30, 17), rng.uniform(-70000, 70000, 100_000)])
    ours = oracle.encode(x, "f16")
    with np.errstate(over="ignore"):
        theirs = x.astype(np.float16).view(np.uint16)
    assert (ours == theirs).all()


def test_encode_f16_halfway_and_overflow():
    # every finite positive fp16 pair (v, next): the midpoint ties to the even pattern
    bits = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = bits.view(np.float16).astype(np.float64)
    hi = (bits + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2  # exact in binary64
    got = oracle.encode(mid, "f16")
    expect = np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16)
    assert (got == expect).all()
    assert (oracle.encode(-mid, "f16") == (expect | 0x8000)).all()
    # just below / at the overflow threshold (65504 + half a quantum of 32)
    assert oracle.encode(np.array([65519.999, 65520.0, 1e300, -65520.0]), "f16").tolist() == \
        [0x7BFF, 0x7C00, 0x7C00, 0xFC00]
    assert oracle.encode(np.array([np.inf, -np.inf, 0.0, -0.0]), "f16").tolist() == \
        [0x7C00, 0xFC00, 0x0000, 0x8000]
    assert oracle.encode(np.array([np.nan]), "f16")[0] & 0x7FFF > 0x7C00
    # subnormal halfway: 2^-25 is halfway between 0 and 2^-24 -> ties to 0 (even)
    assert oracle.encode(np.array([2.0 ** -25, 3 * 2.0 ** -25]), "f16").tolist() == [0x0000, 0x0002]


def test_encode_bf16_against_torch():
    """torch's float32 -> bfloat16 cast is nearest-even; feed values exact in
    float32 so that no double rounding can enter on torch's side."""
    rng = np.random.default_rng(2)
    x32 = np.concatenate([_log_uniform(rng, 400_000, -130, 127),
                          rng.uniform(-3, 3, 100_000)]).astype(np.float32)
    x32 = x32[np.isfinite(x32)]
    ours = oracle.encode(x32.astype(np.float64), "bf16")
    theirs = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (ours == theirs).all()


def test_encode_bf16_halfway_and_overflow():
    bits = np.arange(0, 0x7F7F, 7, dtype=np.uint16)
    dec = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    mid = (dec(bits) + dec(bits + 1)) / 2
    got = oracle.encode(mid, "bf16")
    expect = np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16)
    assert (got == expect).all()
    top = (2 - 2 ** -7) * 2.0 ** 127
    thr = (2 - 2 ** -8) * 2.0 ** 127
    assert oracle.encode(np.array([top, np.nextafter(thr, 0), thr]), "bf16").tolist() == \
        [0x7F7F, 0x7F7F, 0x7F80]


def test_encode_f32_against_numpy():
    rng = np.random.default_rng(3)
    x = np.concatenate([_log_uniform(rng, 300_000, -160, 127), rng.standard_normal(100_000)])
    ours = oracle.encode(x, "f32")
    with np.errstate(over="ignore"):
        theirs = x.astype(np.float32).view(np.uint32)
    assert (ours == theirs).all()


# ------------------------------------------------------------ the product --

def _rand_bits(rng, shape, fmt):
    """Random finite patterns of moderate magnitude (values in about [-2, 2])."""
    v = rng.uniform(-2, 2, shape).astype(np.float32)
    t = torch.from_numpy(v).to(inputs.TORCH_DTYPE[fmt])
    return inputs.to_bits(t)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(1, 1), (3, 8), (5, 7169), (2, 16384), (7, 0), (0, 5)])
def test_ones_closed_form(fmt, n, k):
    """B = ones, a = ones gives c_i = k exactly (and S_i = k)."""
    one = inputs.to_bits(torch.ones(1, dtype=inputs.TORCH_DTYPE[fmt]))[0]
    B = np.full((n, k), one, np.uint16)
    a = np.full((k,), one, np.uint16)
    c, s = oracle.gemv_ref(B, a, fmt)
    assert c.tolist() == [float(k)] * n
    assert s.tolist() == [float(k)] * n


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(6, 10), (10, 6), (9, 9)])
def test_identity_padded(fmt, n, k):
    """B_ij = [i == j]: c_i = a_i for i < min(n, k), else 0.  With n != k this
    also catches a transposed operand or a wrong row stride."""
    rng = np.random.default_rng(n * 100 + k)
    one = inputs.to_bits(torch.ones(1, dtype=inputs.TORCH_DTYPE[fmt]))[0]
    B = np.zeros((n, k), np.uint16)
    for i in range(min(n, k)):
        B[i, i] = one
    a = _rand_bits(rng, (k,), fmt)
    c, _ = oracle.gemv_ref(B, a, fmt)
    a_val = inputs.from_bits(a, fmt).double().numpy()
    expect = np.zeros(n)
    expect[: min(n, k)] = a_val[: min(n, k)]
    assert (c == expect).all()


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_4x8_exact_rationals(fmt, seed):
    """Hand sums of 4x8 inputs in exact rational arithmetic: the binary64
    oracle may differ only by its own rounding, bounded by 7 u S (u = 2^-53)."""
    rng = np.random.default_rng(seed)
    B = _rand_bits(rng, (4, 8), fmt)
    a = _rand_bits(rng, (8,), fmt)
    Bv = inputs.from_bits(B, fmt).double().numpy()
    av = inputs.from_bits(a, fmt).double().numpy()
    c, s = oracle.gemv_ref(B, a, fmt)
    for i in range(4):
        exact = sum(Fraction(float(Bv[i, j])) * Fraction(float(av[j])) for j in range(8))
        S = sum(abs(Fraction(float(Bv[i, j])) * Fraction(float(av[j]))) for j in range(8))
        assert abs(Fraction(c[i]) - exact) <= Fraction(7, 2 ** 53) * S
        assert abs(Fraction(s[i]) - S) <= Fraction(7, 2 ** 53) * S


def test_bruteforce_signs_and_order():
    """A row whose terms cancel exactly: any dropped or sign-flipped term shows."""
    vals = [1.5, -0.25, 3.0, 0.125, -2.0, 0.5, 1.0, -0.75]
    av = [2.0, 4.0, -1.0, 8.0, 0.5, -2.0, 0.25, 1.0]
    B = inputs.to_bits(torch.tensor([vals], dtype=torch.float16))
    a = inputs.to_bits(torch.tensor(av, dtype=torch.float16))
    c, s = oracle.gemv_ref(B, a, "f16")
    exact = sum(Fraction(x) * Fraction(y) for x, y in zip(vals, av))
    assert c[0] == float(exact) == 3.0 - 1.0 - 3.0 + 1.0 - 1.0 - 1.0 + 0.25 - 0.75
    assert s[0] == sum(abs(x * y) for x, y in zip(vals, av))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_numpy_float64_matmul(fmt):
    """numpy's float64 matmul (different summation order) agrees within k u S."""
    rng = np.random.default_rng(7)
    n, k = 48, 777
    B = _rand_bits(rng, (n, k), fmt)
    a = _rand_bits(rng, (k,), fmt)
    c, s = oracle.gemv_ref(B, a, fmt)
    ref = inputs.from_bits(B, fmt).double().numpy() @ inputs.from_bits(a, fmt).double().numpy()
    assert (np.abs(c - ref) <= 2 * k * 2.0 ** -53 * s).all()


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_integer_linearity_and_permutation(fmt):
    """Integer inputs: every partial sum is exact, so c(B, a1 + a2) equals
    c(B, a1) + c(B, a2) exactly, and permuting rows permutes c exactly."""
    n, k = 33, 1001
    B, a1 = inputs.make_int_inputs(n, k, fmt, seed=11)
    _, a2 = inputs.make_int_inputs(1, k, fmt, seed=12)
    Bb, a1b, a2b = inputs.to_bits(B), inputs.to_bits(a1), inputs.to_bits(a2)
    a12 = inputs.to_bits((a1.float() + a2.float()).to(inputs.TORCH_DTYPE[fmt]))
    c1, _ = oracle.gemv_ref(Bb, a1b, fmt)
    c2, _ = oracle.gemv_ref(Bb, a2b, fmt)
    c12, _ = oracle.gemv_ref(Bb, a12, fmt)
    assert (c12 == c1 + c2).all()
    assert (c1 == np.round(c1)).all()
    perm = np.random.default_rng(5).permutation(n)
    cp, _ = oracle.gemv_ref(np.ascontiguousarray(Bb[perm]), a1b, fmt)
    assert (cp == c1[perm]).all()


def test_rows_subset_matches_full():
    rng = np.random.default_rng(9)
    B = _rand_bits(rng, (20, 300), "bf16")
    a = _rand_bits(rng, (300,), "bf16")
    c, s = oracle.gemv_ref(B, a, "bf16")
    rows = np.array([19, 0, 7, 7, 3])
    cr, sr = oracle.gemv_ref_rows(B, a, "bf16", rows)
    assert (cr == c[rows]).all() and (sr == s[rows]).all()
    with pytest.raises(ValueError):
        oracle.gemv_ref_rows(B, a, "bf16", np.array([20]))


def test_nonfinite_stays_in_its_row():
    B = inputs.to_bits(torch.tensor([[1.0, float("inf")], [1.0, 2.0], [float("nan"), 0.0]],
                                    dtype=torch.float16))
    a = inputs.to_bits(torch.tensor([1.0, 1.0], dtype=torch.float16))
    c, _ = oracle.gemv_ref(B, a, "f16")
    assert c[0] == np.inf and c[1] == 3.0 and np.isnan(c[2])


def test_round_out_matches_encode():
    c = np.array([7169.0, 1.0 / 3, -2.5e-8, 70000.0])
    assert oracle.round_out(c, "f16").tolist() == oracle.encode(c, "f16").tolist()
    # k = 7169 rounds to 7168 in fp16 (spacing 4) and in bf16 (spacing 32)
    assert oracle.decode(oracle.round_out(np.array([7169.0]), "f16"), "f16")[0] == 7168.0
    assert oracle.decode(oracle.round_out(np.array([7169.0]), "bf16"), "bf16")[0] == 7168.0


def test_bad_arguments_rejected():
    with pytest.raises(ValueError):
        oracle.gemv_ref(np.zeros((2, 3), np.uint16), np.zeros(4, np.uint16), "f16")
    with pytest.raises(TypeError):
        oracle.gemv_ref(np.zeros((2, 3), np.float32), np.zeros(3, np.uint16), "f16")


# ------------------------------------------------------ acceptance rules --

def test_case_a_error_table_is_flagged():
    """The errors the pages print for their broken design are flagged as a
    power-of-two pattern by the acceptance rules, for either output format."""
    rows = _golden_rows("case_a_max_err.txt")
    errs = np.array([float(r[3]) for r in rows])
    assert errs.tolist() == [0.125, 0.125, 0.125, 0.25]
    c_ref = np.full(errs.shape, 3.3)
    for fmt in ("f16", "bf16", "f32"):
        assert parity_rules.pow2_errors(errs, c_ref, fmt).all()
        with pytest.raises(AssertionError, match="power-of-two"):
            # reported as the design-bug signature before any tolerance test
            # (for fp32 output with this S the tolerance alone would pass them)
            parity_rules.check(3.3 + errs, c_ref, np.full(errs.shape, 1e9), fmt)
    # rounding-sized errors are not flagged
    assert not parity_rules.pow2_errors(np.array([2.0 ** -9]), np.array([3.3]), "f16").any()


def test_acceptance_tolerances():
    c_ref = np.array([0.5, 100.0, -3.0])
    parity_rules.check(c_ref + np.array([0.009, 0.9, -0.02]), c_ref, np.ones(3), "f16")
    with pytest.raises(AssertionError):
        parity_rules.check(c_ref + np.array([0.011, 0.0, 0.0]), c_ref, np.ones(3), "bf16")
    s = np.array([1000.0, 1000.0, 1000.0])
    parity_rules.check(c_ref + 0.009, c_ref, s, "f32")
    with pytest.raises(AssertionError):
        parity_rules.check(c_ref + 0.011, c_ref, s, "f32")
    with pytest.raises(AssertionError):
        parity_rules.check(np.array([np.inf]), np.array([np.nan]), np.ones(1), "f16")


def test_ulp_helper():
    assert parity_rules.ulp(np.array([1.0, 1.5, 2.0, 0.0]), "f16").tolist() == \
        [2.0 ** -10, 2.0 ** -10, 2.0 ** -9, 2.0 ** -24]
    assert parity_rules.ulp(np.array([7168.0]), "bf16")[0] == 32.0
    assert math.isclose(parity_rules.ulp(np.array([1.0]), "f32")[0], 2.0 ** -23)


# ------------------------------------------------------------- epilogue --

def test_epilogue_closed_forms():
    """Values the activations' definitions fix exactly (or to one rounding)."""
    ln3 = math.log(3.0)
    c = np.array([0.0, ln3, -ln3, 2.5, -2.5, 0.0])
    s = np.abs(c)
    y, _ = oracle.gemv_ref_epilogue(c, s, act="sigmoid")
    assert y[0] == 0.5
    assert abs(y[1] - 0.75) <= 2 ** -52 and abs(y[2] - 0.25) <= 2 ** -53
    assert abs(y[3] + y[4] - 1.0) <= 2 ** -52  # sigmoid(x) + sigmoid(-x) = 1
    y, _ = oracle.gemv_ref_epilogue(c, s, act="silu")
    assert y[0] == 0.0 and abs(y[1] - 0.75 * ln3) <= 2 ** -51
    assert abs((y[3] - y[4]) - 2.5) <= 2 ** -50  # silu(x) - silu(-x) = x
    y, _ = oracle.gemv_ref_epilogue(c, s, act="relu")
    assert y.tolist() == [0.0, ln3, 0.0, 2.5, 0.0, 0.0]
    nan_y, _ = oracle.gemv_ref_epilogue(np.array([np.nan]), np.array([0.0]), act="relu")
    assert nan_y[0] == 0.0  # max(NaN, 0) taken as 0


def test_epilogue_scale_and_bias_exact():
    """Identity activation: y = alpha c + beta bias exactly for small dyadic
    values, with the bias decoded from each format's bit patterns."""
    c = np.array([1.0, -2.0, 0.5, 3.0])
    s = np.array([4.0, 2.0, 1.0, 3.0])
    bias = np.array([0.25, -1.0, 8.0, 0.0])
    for fmt, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        bits = inputs.to_bits(torch.tensor(bias, dtype=tdt))
        y, scale = oracle.gemv_ref_epilogue(c, s, alpha=2.0, beta=-0.5, bias_bits=bits, bias_fmt=fmt)
        assert y.tolist() == (2.0 * c - 0.5 * bias).tolist()
        assert scale.tolist() == (2.0 * s + 0.5 * np.abs(bias)).tolist()
    bits32 = bias.astype(np.float32).view(np.uint32)
    y, _ = oracle.gemv_ref_epilogue(c, s, alpha=1.0, beta=1.0, bias_bits=bits32, bias_fmt="f32")
    assert y.tolist() == (c + bias).tolist()
    y, scale = oracle.gemv_ref_epilogue(c, s)  # defaults: identity
    assert y.tolist() == c.tolist() and scale.tolist() == s.tolist()
    _, scale = oracle.gemv_ref_epilogue(c, s, act="sigmoid")
    assert scale.tolist() == (0.25 * s).tolist()

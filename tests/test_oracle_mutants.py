"""Planted mistakes in a copy of the oracle must be caught by the pins.

Each mutant is the oracle's C source with one plausible slip (a dropped term,
a flipped sign, a transposed operand, a wrong exponent bias, truncating ties,
...) compiled into a temporary library.  The pin checks below (the same
external facts test_oracle.py uses: torch/numpy casts, closed forms, exact
rational sums) are run against it; at least one must fail.  The real oracle
must pass all of them.  CPU only; the mutants never touch a GPU.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from memory_bound_gemv_02_gb300 import inputs

MUTANTS = {
    "dropped_last_term": ("for (int64_t j = 0; j < k; ++j) {", "for (int64_t j = 0; j + 1 < k; ++j) {"),
    "dropped_first_term": ("for (int64_t j = 0; j < k; ++j) {", "for (int64_t j = 1; j < k; ++j) {"),
    "sign_flip": ("      acc += p;", "      acc -= p;"),
    "transposed_B": ("B[i * k + j]", "B[i + j * n]"),
    "reversed_a": ("* ref_decode_bits(a[j], in_fmt)", "* ref_decode_bits(a[k - 1 - j], in_fmt)"),
    "row_stride": ("B[i * k + j]", "B[i * (k - (k > 1)) + j]"),
    "bias_off_by_one": ("const int bias = (1 << (ebits - 1)) - 1;\n  const uint32_t emax_field = (1u << ebits) - 1u;\n  const uint32_t sign = (bits",
                        "const int bias = (1 << (ebits - 1));\n  const uint32_t emax_field = (1u << ebits) - 1u;\n  const uint32_t sign = (bits"),
    "subnormal_scale": ("v = ldexp((double)m, 1 - bias - mbits);", "v = ldexp((double)m, -bias - mbits);"),
    "ties_truncate": ("r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "r = fl;"),
    "ties_away": ("r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "r = fl + 1.0;"),
    "abs_sum_signed": ("acc_abs += fabs(p);", "acc_abs += p;"),
    "bf16_as_f16": ("if (fmt == REF_F16) {", "if (fmt == REF_F16 || fmt == REF_BF16) {"),
    "sigmoid_sign": ("case REF_ACT_SIGMOID: return 1.0 / (1.0 + exp(-y));", "case REF_ACT_SIGMOID: return 1.0 / (1.0 + exp(y));"),
    "silu_as_sigmoid": ("case REF_ACT_SILU: return y / (1.0 + exp(-y));", "case REF_ACT_SILU: return 1.0 / (1.0 + exp(-y));"),
    "bias_sign": ("double pre = alpha * c[i] + beta * b;", "double pre = alpha * c[i] - beta * b;"),
    "relu_leaky": ("case REF_ACT_RELU: return y > 0.0 ? y : 0.0;", "case REF_ACT_RELU: return y > 0.0 ? y : 0.01 * y;"),
    "gla_decay_on_kv": ("const double sn = decay * sij + kv;", "const double sn = sij + decay * kv;"),
    "gla_no_scale": ("o[h * dv + j] = scale * acc;", "o[h * dv + j] = acc;"),
    "gla_transposed_state": ("ref_load(S, (h * dk + i) * dv + j, fmt)", "ref_load(S, (h * dv + j) * dk + i, fmt)"),
    "gla_o_from_old_state": ("acc += qi * sn;", "acc += qi * sij;"),
    "gla_decay_sign": ("const double decay = exp(ref_load(gk, h * dk + i, fmt));",
                       "const double decay = exp(-ref_load(gk, h * dk + i, fmt));"),
    "gla_q_for_k": ("const double kv = ref_load(k, h * dk + i, fmt)", "const double kv = ref_load(q, h * dk + i, fmt)"),
    "gla_v_head_stride": ("ref_load(v, h * dv + j, fmt)", "ref_load(v, h * dk + j, fmt)"),
    "gla_abs_sum_merged": ("ss[(h * dk + i) * dv + j] = fabs(decay * sij) + fabs(kv);",
                           "ss[(h * dk + i) * dv + j] = fabs(decay * sij + kv);"),
    "gla_abs_o_signed": ("acc_abs += fabs(qi * sn);", "acc_abs += qi * sn;"),
}


def _check_decode(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for fmt, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        ours = o.decode(bits, fmt)
        theirs = torch.from_numpy(bits.view(np.int16).copy()).view(tdt).double().numpy()
        m = ~np.isnan(theirs)
        assert (ours[m] == theirs[m]).all()


def _check_encode(o):
    rng = np.random.default_rng(1)
    x = np.exp2(rng.uniform(-30, 17, 20000)) * np.where(rng.random(20000) < 0.5, -1, 1)
    with np.errstate(over="ignore"):
        assert (o.encode(x, "f16") == x.astype(np.float16).view(np.uint16)).all()
    bits = np.arange(0, 0x7BFF, dtype=np.uint16)
    mid = (bits.view(np.float16).astype(np.float64) + (bits + 1).view(np.float16).astype(np.float64)) / 2
    assert (o.encode(mid, "f16") == np.where(bits % 2 == 0, bits, bits + 1)).all()


def _check_closed_forms(o):
    for fmt in ("f16", "bf16"):
        one = inputs.to_bits(torch.ones(1, dtype=inputs.TORCH_DTYPE[fmt]))[0]
        for n, k in ((3, 8), (5, 77)):
            c, s = o.gemv_ref(np.full((n, k), one, np.uint16), np.full(k, one, np.uint16), fmt)
            assert c.tolist() == [float(k)] * n and s.tolist() == [float(k)] * n
        for n, k in ((6, 10), (10, 6)):
            rng = np.random.default_rng(n + k)
            B = np.zeros((n, k), np.uint16)
            for i in range(min(n, k)):
                B[i, i] = one
            a = inputs.to_bits(torch.from_numpy(rng.uniform(-2, 2, k).astype(np.float32))
                               .to(inputs.TORCH_DTYPE[fmt]))
            c, _ = o.gemv_ref(B, a, fmt)
            expect = np.zeros(n)
            expect[: min(n, k)] = inputs.from_bits(a, fmt).double().numpy()[: min(n, k)]
            assert (c == expect).all()


def _check_bruteforce(o):
    for fmt in ("f16", "bf16"):
        for seed in range(3):
            rng = np.random.default_rng(seed)
            tdt = inputs.TORCH_DTYPE[fmt]
            B = inputs.to_bits(torch.from_numpy(rng.uniform(-2, 2, (4, 8)).astype(np.float32)).to(tdt))
            a = inputs.to_bits(torch.from_numpy(rng.uniform(-2, 2, 8).astype(np.float32)).to(tdt))
            Bv = inputs.from_bits(B, fmt).double().numpy()
            av = inputs.from_bits(a, fmt).double().numpy()
            c, s = o.gemv_ref(B, a, fmt)
            for i in range(4):
                terms = [Fraction(float(Bv[i, j])) * Fraction(float(av[j])) for j in range(8)]
                S = sum(abs(t) for t in terms)
                assert abs(Fraction(c[i]) - sum(terms)) <= Fraction(7, 2 ** 53) * S
                assert abs(Fraction(s[i]) - S) <= Fraction(7, 2 ** 53) * S


def _check_epilogue(o):
    ln3 = math.log(3.0)
    c = np.array([0.0, ln3, -2.0, 2.5])
    s = np.abs(c)
    y, _ = o.gemv_ref_epilogue(c, s, act="sigmoid")
    assert y[0] == 0.5 and abs(y[1] - 0.75) <= 2 ** -52
    y, _ = o.gemv_ref_epilogue(c, s, act="silu")
    assert abs(y[1] - 0.75 * ln3) <= 2 ** -51
    y, _ = o.gemv_ref_epilogue(c, s, act="relu")
    assert y.tolist() == [0.0, ln3, 0.0, 2.5]
    bits = inputs.to_bits(torch.tensor([1.0, 2.0, 3.0, 4.0], dtype=torch.float16))
    y, _ = o.gemv_ref_epilogue(c, s, alpha=2.0, beta=0.5, bias_bits=bits, bias_fmt="f16")
    assert y.tolist() == (2.0 * c + 0.5 * np.array([1.0, 2.0, 3.0, 4.0])).tolist()


def _check_gla(o):
    def bits(x):
        return np.asarray(x, dtype=np.float32).view(np.uint32)
    rng = np.random.default_rng(3)
    bh, dk, dv = 2, 3, 5
    q = rng.integers(-3, 4, (bh, dk)).astype(np.float64)
    k = rng.integers(-3, 4, (bh, dk)).astype(np.float64)
    v = rng.integers(-3, 4, (bh, dv)).astype(np.float64)
    S = rng.integers(-3, 4, (bh, dk, dv)).astype(np.float64)
    for gk_val, decay in ((0.0, 1.0), (-np.inf, 0.0)):
        gk = np.full((bh, dk), gk_val)
        S_new, out, ss, os_ = o.gla_ref_decode(bits(q), bits(k), bits(v), bits(gk), bits(S), 0.5, "f32")
        kv = k[:, :, None] * v[:, None, :]
        want = decay * S + kv
        assert (S_new == want).all()
        assert (out == 0.5 * np.einsum("hi,hij->hj", q, want)).all()
        # the magnitudes behind the tolerances, exact for these integers
        assert (ss == np.abs(decay * S) + np.abs(kv)).all()
        assert (os_ == 0.5 * np.einsum("hi,hij->hj", np.abs(q), np.abs(want))).all()


PINS = [_check_decode, _check_encode, _check_closed_forms, _check_bruteforce, _check_epilogue, _check_gla]


def _failures(o):
    failed = []
    for pin in PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


def test_real_oracle_passes_every_pin():
    assert _failures(oracle.default()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    failed = _failures(oracle.Oracle(lib))
    assert failed, f"mutant {name} passed every pin"

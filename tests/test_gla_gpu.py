"""GLA decode step on the GPU (gla_decode) against the oracle.

S_new = diag(exp(gk)) S + outer(k, v), o = scale * q^T S_new per head
(TileLang Case Studies, Case D "Background").  The kernel works in fp32 and
rounds each stored value once; the oracle works in binary64.

Tolerances, from the arithmetic: an S_new element is fmaf(exp(gk), S,
k*v) -- a few fp32 roundings plus expf's error, within 8 u32 of
|exp(gk) S| + |k v| -- then rounded once to the storage type (half an ulp).
o sums dk fp32 products: within 1e-5 * |scale| sum |q S_new| plus the S_new
errors it carries (|scale| sum |q| 8 u32 (|exp(gk) S| + |k v|)), then rounded
to the storage type.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import kernel_model
import memory_bound_gemv_02_gb300 as g
import oracle
import parity_rules

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24
FMT = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}


def _bits(t):
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


def _make(bh, dk, dv, dtype, seed, dev):
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)

    def u(*shape, lo=-1.0, hi=1.0):
        return (torch.rand(shape, generator=gen, device=dev) * (hi - lo) + lo).to(dtype)
    q, k, v = u(bh, dk), u(bh, dk), u(bh, dv)
    gk = u(bh, dk, lo=-3.0, hi=0.0)
    S = (torch.randn((bh, dk, dv), generator=gen, device=dev)).to(dtype)
    return q, k, v, gk, S


def _check(q, k, v, gk, S_in, S_new, o, scale, label):
    torch.cuda.synchronize()
    fmt = FMT[S_in.dtype]
    ref_S, ref_o, ss, os_ = oracle.gla_ref_decode(_bits(q), _bits(k), _bits(v), _bits(gk), _bits(S_in), scale, fmt)
    got_S = S_new.double().cpu().numpy()
    got_o = o.double().cpu().numpy()
    tol_S = 8 * U32 * ss + (0 if fmt == "f32" else 0.5) * parity_rules.ulp(ref_S, fmt)
    # o inherits the fp32 error of each S_new element it sums (which is
    # relative to |exp(gk) S| + |k v|, not to |S_new|) plus its own sum's.
    qd = q.double().cpu().numpy()
    carried = abs(scale) * np.einsum("hi,hij->hj", np.abs(qd), 8 * U32 * ss)
    tol_o = 1e-5 * os_ + carried + (0 if fmt == "f32" else 0.5) * parity_rules.ulp(ref_o, fmt) + 1e-30
    bad_S = ~(np.abs(got_S - ref_S) <= tol_S)
    bad_o = ~(np.abs(got_o - ref_o) <= tol_o)
    assert not bad_S.any(), f"{label}: S_new off at {np.argwhere(bad_S)[:4].tolist()}"
    assert not bad_o.any(), f"{label}: o off at {np.argwhere(bad_o)[:4].tolist()}"
    for err, ref in ((got_S - ref_S, ref_S), (got_o - ref_o, ref_o)):
        assert not parity_rules.pow2_errors(err, ref, fmt).any(), f"{label}: power-of-two error pattern"


SHAPES = [(64, 128, 128), (32, 64, 64), (8, 256, 128), (3, 17, 8), (2, 1, 512), (4, 100, 1024), (1, 4096, 64)]


def _warp_ok(dv, dtype):
    """One warp per head needs dv * element size <= 512 bytes."""
    return dv * (4 if dtype == torch.float32 else 2) <= 512


def _pipe_ok(dk, dv, dtype):
    """The pipelined layout's shape condition (pointers 16-byte aligned)."""
    return kernel_model.gla_pipe_ok(dk, dv, 4 if dtype == torch.float32 else 2)


def _variant_ok(variant, dk, dv, dtype):
    if variant == g.GLA_VARIANT_WARP:
        return _warp_ok(dv, dtype)
    if variant == g.GLA_VARIANT_PIPE:
        return _pipe_ok(dk, dv, dtype)
    return True


ALL = [g.GLA_VARIANT_AUTO, g.GLA_VARIANT_CTA, g.GLA_VARIANT_WARP, g.GLA_VARIANT_PIPE]
FORCED = [g.GLA_VARIANT_CTA, g.GLA_VARIANT_WARP, g.GLA_VARIANT_PIPE]


@pytest.mark.parametrize("bh,dk,dv", SHAPES + [(40, 64, 64), (9, 33, 256), (37, 16, 64), (11, 5, 24), (300, 8, 64)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("variant", ALL)
def test_gla_parity(cuda_dev, bh, dk, dv, dtype, variant):
    if dtype == torch.float32 and dv // 4 > 256:
        pytest.skip("dv / 4 > 256 is outside the kernel's range for fp32")
    if not _variant_ok(variant, dk, dv, dtype):
        with pytest.raises(g.GemvError) as ei:
            q, k, v, gk, S = _make(bh, dk, dv, dtype, 1, cuda_dev)
            g.gla_decode(q, k, v, gk, S, scale=1.0, variant=variant)
        assert ei.value.status == g.GEMV_ERR_CONFIG
        return
    q, k, v, gk, S = _make(bh, dk, dv, dtype, bh + dk + dv, cuda_dev)
    S_in = S.clone()
    S_new, o = g.gla_decode(q, k, v, gk, S, scale=dk ** -0.5, variant=variant)
    _check(q, k, v, gk, S_in, S_new, o, dk ** -0.5, f"{bh}x{dk}x{dv} {dtype} variant {variant}")
    assert torch.equal(S, S_in)  # out of place: S untouched


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("variant", FORCED)
def test_gla_in_place(cuda_dev, dtype, variant):
    d = 64 if dtype == torch.float32 else 128  # a shape every layout takes
    q, k, v, gk, S = _make(16, d, d, dtype, 5, cuda_dev)
    S_in = S.clone()
    S_new, o = g.gla_decode(q, k, v, gk, S, scale=0.125, S_new=S, variant=variant)
    assert S_new.data_ptr() == S.data_ptr()
    _check(q, k, v, gk, S_in, S_new, o, 0.125, f"in place {dtype} variant {variant}")


@pytest.mark.parametrize("bh,dk,dv,dtype", [(4096, 64, 64, torch.float16), (2600, 128, 128, torch.bfloat16),
                                            (3000, 16, 128, torch.float32), (5, 200, 40, torch.float16)])
def test_gla_layouts_agree(cuda_dev, bh, dk, dv, dtype):
    """The layouts store bit-identical states (same fmaf per element) and o
    within the sum-order tolerance; the automatic choice is the pipelined
    layout where it applies, else the CTA layout."""
    q, k, v, gk, S = _make(bh, dk, dv, dtype, 21, cuda_dev)
    S_c, o_c = g.gla_decode(q, k, v, gk, S, scale=0.25, variant=g.GLA_VARIANT_CTA)
    S_w, o_w = g.gla_decode(q, k, v, gk, S, scale=0.25, variant=g.GLA_VARIANT_WARP)
    outs = {"cta": (S_c, o_c), "warp": (S_w, o_w)}
    pipe = _pipe_ok(dk, dv, dtype)
    if pipe:
        outs["pipe"] = g.gla_decode(q, k, v, gk, S, scale=0.25, variant=g.GLA_VARIANT_PIPE)
    torch.cuda.synchronize()
    for name, (S_x, o_x) in outs.items():
        assert torch.equal(_t(S_c), _t(S_x)), name
        if bh <= 64:
            _check(q, k, v, gk, S, S_x, o_x, 0.25, f"{name} layout")
        else:
            rows = torch.arange(0, bh, max(1, bh // 40), device=cuda_dev)
            _check(q[rows], k[rows], v[rows], gk[rows], S[rows], S_x[rows], o_x[rows], 0.25, f"{name} sampled")
    S_a, o_a = g.gla_decode(q, k, v, gk, S, scale=0.25)
    torch.cuda.synchronize()
    want = outs["pipe" if kernel_model.gla_auto_is_pipe(dk, dv, 4 if dtype == torch.float32 else 2) else "cta"]
    assert torch.equal(_t(o_a), _t(want[1])) and torch.equal(_t(S_a), _t(want[0]))


@pytest.mark.parametrize("bh,dk,dv,dtype", [(2048, 128, 128, torch.bfloat16), (300, 64, 128, torch.float32),
                                            (37, 32, 256, torch.float16), (1000, 8, 16, torch.bfloat16)])
def test_gla_pipe_same_heads_per_round_bit_identical(cuda_dev, bh, dk, dv, dtype):
    """Where the pipelined and the CTA layouts take the same heads per round
    (G), they sum o in the same row blocks in the same order: both outputs
    are bit-identical."""
    es = 4 if dtype == torch.float32 else 2
    cpr = dv * es // 16
    G_pipe = kernel_model.gla_pipe_heads_per_cta(bh, dk, dv, es)
    G_cta = kernel_model.gla_heads_per_cta(bh, dk, cpr)
    if G_pipe != G_cta:
        pytest.skip(f"heads per round differ ({G_pipe} vs {G_cta})")
    q, k, v, gk, S = _make(bh, dk, dv, dtype, 23, cuda_dev)
    S_c, o_c = g.gla_decode(q, k, v, gk, S, scale=0.3, variant=g.GLA_VARIANT_CTA)
    S_p, o_p = g.gla_decode(q, k, v, gk, S, scale=0.3, variant=g.GLA_VARIANT_PIPE)
    torch.cuda.synchronize()
    assert torch.equal(_t(S_c), _t(S_p)) and torch.equal(_t(o_c), _t(o_p))


def test_gla_pipe_alignment_fallback(cuda_dev):
    """q one element off a 16-byte boundary: the automatic choice falls back
    to the CTA layout (same results), the pipelined layout refuses."""
    bh, dk, dv = 64, 64, 64
    q, k, v, gk, S = _make(bh, dk, dv, torch.float16, 24, cuda_dev)
    qbuf = torch.empty(bh * dk + 1, dtype=torch.float16, device=cuda_dev)
    qbuf[1:].copy_(q.reshape(-1))
    q_off = qbuf[1:].view(bh, dk)
    S_a, o_a = g.gla_decode(q_off, k, v, gk, S, scale=0.2)
    S_c, o_c = g.gla_decode(q, k, v, gk, S, scale=0.2, variant=g.GLA_VARIANT_CTA)
    torch.cuda.synchronize()
    assert torch.equal(_t(S_a), _t(S_c)) and torch.equal(_t(o_a), _t(o_c))
    with pytest.raises(g.GemvError) as ei:
        g.gla_decode(q_off, k, v, gk, S, scale=0.2, variant=g.GLA_VARIANT_PIPE)
    assert ei.value.status == g.GEMV_ERR_CONFIG


def _t(x):
    return x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("variant", FORCED)
def test_gla_integer_inputs_no_decay_exact(cuda_dev, dtype, variant):
    """gk = 0 and small integers: every fp32 operation is exact, so the stored
    state and o equal the oracle rounded once."""
    gen = torch.Generator(device=cuda_dev)
    gen.manual_seed(3)
    bh, dk, dv = 8, 64, 128
    ri = lambda *s: torch.randint(-3, 4, s, generator=gen, device=cuda_dev).to(dtype)
    q, k, v, S = ri(bh, dk), ri(bh, dk), ri(bh, dv), ri(bh, dk, dv)
    gk = torch.zeros((bh, dk), dtype=dtype, device=cuda_dev)
    S_new, o = g.gla_decode(q, k, v, gk, S, scale=0.5, variant=variant)
    torch.cuda.synchronize()
    fmt = FMT[dtype]
    ref_S, ref_o, _, _ = oracle.gla_ref_decode(_bits(q), _bits(k), _bits(v), _bits(gk), _bits(S), 0.5, fmt)
    assert (_bits(S_new) == oracle.encode(ref_S, fmt)).all()
    assert (_bits(o) == oracle.encode(ref_o, fmt)).all()


@pytest.mark.parametrize("variant", FORCED)
def test_gla_multiple_steps_match_stepwise_oracle(cuda_dev, variant):
    """Ten chained decode steps on one state (in place), each checked."""
    bh, dk, dv = 12, 64, 64
    q, k, v, gk, S = _make(bh, dk, dv, torch.float32, 9, cuda_dev)
    for step in range(10):
        q, k, v, gk, _ = _make(bh, dk, dv, torch.float32, 100 + step, cuda_dev)
        S_prev = S.clone()
        _, o = g.gla_decode(q, k, v, gk, S, scale=0.1, S_new=S, variant=variant)
        _check(q, k, v, gk, S_prev, S, o, 0.1, f"step {step}")


def test_gla_empty_dk_and_errors(cuda_dev):
    bh, dv = 3, 64
    z = torch.empty((bh, 0), dtype=torch.bfloat16, device=cuda_dev)
    S = torch.empty((bh, 0, dv), dtype=torch.bfloat16, device=cuda_dev)
    v = torch.ones((bh, dv), dtype=torch.bfloat16, device=cuda_dev)
    o = torch.full((bh, dv), 7.0, dtype=torch.bfloat16, device=cuda_dev)
    g.gla_decode(z, z, v, z, S, scale=1.0, o=o)
    torch.cuda.synchronize()
    assert (o == 0).all()
    q, k, v, gk, S = _make(2, 16, 24, torch.bfloat16, 1, cuda_dev)
    with pytest.raises(g.GemvError) as ei:
        g.gla_decode(q, k, v, gk, S, scale=1.0)  # dv = 24 is a multiple of 8: fine
        g.gla_decode(q, k, v[:, :20].contiguous(), gk, S[:, :, :20].contiguous(), scale=1.0)  # 20 % 8 != 0
    assert ei.value.status == g.GEMV_ERR_ARG
    base = torch.zeros(2 * 16 * 32 + 8, dtype=torch.bfloat16, device=cuda_dev)
    S0 = base[:2 * 16 * 32].view(2, 16, 32)
    S1 = base[8:8 + 2 * 16 * 32].view(2, 16, 32)  # 16 bytes further: overlaps S0, is not S0
    with pytest.raises(g.GemvError) as ei:
        g.gla_decode(q, k, torch.zeros((2, 32), dtype=torch.bfloat16, device=cuda_dev), gk, S0, scale=1.0,
                     S_new=S1)
    assert ei.value.status == g.GEMV_ERR_ALIAS


@pytest.mark.parametrize("variant", ALL)
@pytest.mark.parametrize("bh,d,dtype", [(64, 64, torch.bfloat16), (300, 128, torch.float16), (48, 32, torch.float32)])
def test_gla_prefetch_state_layer_chain(cuda_dev, variant, bh, d, dtype):
    """GLA_PREFETCH_STATE over a stack of layers, each owning its state: step
    t of layer l follows step t of layer l-1 on the stream and reads that
    step's o as its v, so only the state may be requested before the wait.
    An ordinary kernel separates one step's layers from the next step's (the
    promise's condition: the last write of a layer's state has completed).
    Every step is checked against the oracle on the values it read."""
    layers, steps, scale = 4, 3, d ** -0.5
    states = [_make(bh, d, d, dtype, 40 + l, cuda_dev)[4] for l in range(layers)]
    for t in range(steps):
        _, _, v, _, _ = _make(bh, d, d, dtype, 200 + t, cuda_dev)
        for l in range(layers):
            q, k, _, gk, _ = _make(bh, d, d, dtype, 300 + 10 * t + l, cuda_dev)
            S_prev = states[l].clone()
            _, o = g.gla_decode(q, k, v, gk, states[l], scale=scale, S_new=states[l], variant=variant,
                                flags=g.GLA_PREFETCH_STATE)
            _check(q, k, v, gk, S_prev, states[l], o, scale, f"step {t} layer {l}")
            v = o
    # without the checks in between: the same chain back to back, compared
    # with a run that waits before every access
    for flags in (g.GLA_PREFETCH_STATE, 0):
        st = [_make(bh, d, d, dtype, 40 + l, cuda_dev)[4] for l in range(layers)]
        ins = [_make(bh, d, d, dtype, 500 + l, cuda_dev) for l in range(layers)]
        v = ins[0][2]
        for t in range(steps):
            v = v * 1  # an ordinary launch between steps
            for l in range(layers):
                q, k, _, gk, _ = ins[l]
                _, v = g.gla_decode(q, k, v, gk, st[l], scale=scale, S_new=st[l], variant=variant, flags=flags)
        torch.cuda.synchronize()
        if flags:
            want = (v.clone(), [x.clone() for x in st])
    assert torch.equal(_t(v), _t(want[0])) and all(torch.equal(_t(a), _t(b)) for a, b in zip(st, want[1]))


def test_gla_flags_rejected(cuda_dev):
    q, k, v, gk, S = _make(2, 16, 24, torch.bfloat16, 1, cuda_dev)
    for bad in (2, 1 << 8, -1):
        with pytest.raises(g.GemvError) as ei:
            g.gla_decode(q, k, v, gk, S, scale=1.0, flags=bad)
        assert ei.value.status == g.GEMV_ERR_ARG

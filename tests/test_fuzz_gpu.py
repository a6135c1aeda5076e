"""Seeded random cases through the GEMV and GLA entry points on the GPU.

Each GEMV case draws a shape, a pointer offset of B, a row stride, the input
and output types, a forced launch configuration (or none) and an epilogue
(or none).  Before anything is launched, the configuration the library will
use is replayed on the CPU by the kernel model (every block read inside B,
every element covered once, every ring chunk in its buffer); then the result
is compared with the oracle under the same tolerances as every other parity
test (16-bit output 1e-2 * max(1, |c_ref|); fp32 output 1e-5 * sum |B a|,
widened for the epilogue by its slope and its own fp32 rounding; the
power-of-two rule).  GLA cases likewise replay the chosen layout first.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import kernel_model
import memory_bound_gemv_02_gb300 as g
import oracle
import parity_rules
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu

NS = [1, 2, 7, 31, 64, 97, 256, 513, 1000, 2048, 3001]
KS = [1, 3, 8, 17, 64, 100, 513, 1031, 4096, 4099, 7169, 16384, 33000]
CONFIGS = [None, {"variant": 3}, {"variant": 4}, {"variant": 2}, {"grid_split": 3}, {"warp_split": 2},
           {"variant": 4, "stages": 3}, {"overlap": 2}, {"overlap": 0}, {"variant": 3, "rows_per_warp": 2, "unroll": 4},
           {"variant": 4, "warp_split": 4, "overlap": 3}, {"overlap": 3}, {"variant": 3, "warp_split": 2, "overlap": 3}]
ACTS = [None, None, "relu", "sigmoid", "silu"]
SLOPE = {None: 1.0, "none": 1.0, "relu": 1.0, "sigmoid": 0.25, "silu": 1.1}


def _draw(rng):
    return dict(n=int(rng.choice(NS)), k=int(rng.choice(KS)), dtype=str(rng.choice(["f16", "bf16"])),
                out_fp32=bool(rng.integers(2)), b_off=int(rng.choice([0, 0, 1, 3, 7])),
                pad=int(rng.choice([0, 0, 1, 8, 13])), cfg=CONFIGS[int(rng.integers(len(CONFIGS)))],
                act=ACTS[int(rng.integers(len(ACTS)))], seed=int(rng.integers(1 << 30)))


@pytest.mark.parametrize("case", range(120))
def test_gemv_fuzz(cuda_dev, case):
    p = _draw(np.random.default_rng(1000 + case))
    n, k, dtype, out_fp32, b_off, pad, cfg, act = (p[x] for x in ("n", "k", "dtype", "out_fp32", "b_off", "pad",
                                                                   "cfg", "act"))
    ldb = k + pad
    if cfg and cfg.get("variant") == 2 and pad:
        pad, ldb = 0, k  # the CPU model of the row-per-warp kernel covers dense rows only
    td = inputs.TORCH_DTYPE[dtype]
    aligned = b_off == 0 and ldb % 8 == 0
    # the launch the library will make, replayed on the CPU first
    try:
        plan = g.gemv_plan(n, k, g.dtype_code(td, out_fp32), aligned,
                           torch.cuda.get_device_properties(cuda_dev).multi_processor_count, config=cfg)
    except g.GemvError as e:
        assert e.status == g.GEMV_ERR_CONFIG
        return
    if n * k <= 30_000_000:  # larger plans are replayed in full by the CPU suite's workload-shape tests
        kernel_model.replay(n, k, plan, base_off=b_off, ldb=ldb)

    Bc, a = inputs.make_inputs(n, k, dtype, "uniform", p["seed"], cuda_dev)
    buf = torch.full((b_off + n * ldb + 8,), float("nan"), dtype=td, device=cuda_dev)
    Bv = buf[b_off:b_off + n * ldb].view(n, ldb)[:, :k]
    Bv.copy_(Bc)
    bias = None
    if act is not None:
        bias = (torch.rand(n, generator=inputs.generator(p["seed"] + 1, cuda_dev), device=cuda_dev) * 2 - 1)
    if act is None and pad == 0:
        c = g.gemv_ex(Bv, a, out_fp32=out_fp32, config=cfg)
    else:
        c = g.gemv_fused(Bv, a, out_fp32=out_fp32, alpha=0.75, beta=0.5 if bias is not None else 0.0, bias=bias,
                         activation=act or "none", config=cfg)
    used = g.gemv_last_config()
    assert {kk: used[kk] for kk in ("variant", "warp_split", "rows_per_warp", "grid_split", "ctas")} == \
        {kk: plan[kk] for kk in ("variant", "warp_split", "rows_per_warp", "grid_split", "ctas")}
    torch.cuda.synchronize()

    c_ref, s_ref = oracle.gemv_ref(inputs.to_bits(Bc), inputs.to_bits(a), dtype)
    alpha, beta = (1.0, 0.0) if (act is None and pad == 0) else (0.75, 0.5 if bias is not None else 0.0)
    bias_bits = None if bias is None else bias.cpu().numpy().view(np.uint32)
    y_ref, scale = oracle.gemv_ref_epilogue(c_ref, s_ref, alpha, beta, bias_bits, "f32", act or "none")
    got = c.double().cpu().numpy()
    out_fmt = "f32" if out_fp32 else dtype
    if out_fp32:
        tol = 1e-5 * scale * SLOPE[act] + 2e-6 * np.abs(y_ref) + 1e-30
    else:
        tol = 1e-2 * np.maximum(1.0, np.abs(y_ref))
    err = got - y_ref
    label = f"case {case}: {p} plan {plan}"
    assert not parity_rules.pow2_errors(err, y_ref, out_fmt).any(), f"{label}: power-of-two errors"
    bad = ~(np.abs(err) <= tol)
    assert not bad.any(), f"{label}: {int(bad.sum())} rows off, first {np.flatnonzero(bad)[:5]}"
    # the stride padding (NaN) and the guard elements are untouched inputs: nothing wrote into B
    assert torch.isnan(buf[:b_off]).all() and torch.isnan(buf[b_off + n * ldb:]).all()


@pytest.mark.parametrize("case", range(40))
def test_gla_fuzz(cuda_dev, case):
    rng = np.random.default_rng(5000 + case)
    dt = [torch.float16, torch.bfloat16, torch.float32][int(rng.integers(3))]
    es = 4 if dt == torch.float32 else 2
    vec = 16 // es
    bh = int(rng.choice([1, 3, 17, 64, 300]))
    dk = int(rng.choice([0, 1, 5, 16, 64, 100, 128, 256]))
    dv = vec * int(rng.choice([1, 2, 3, 5, 8, 16, 32]))
    variant = int(rng.choice([0, 1, 2, 3]))
    in_place = bool(rng.integers(2))
    warp_ok = dv * es <= 512
    pipe_ok = kernel_model.gla_pipe_ok(dk, dv, es)
    if (variant == 2 and not warp_ok) or (variant == 3 and not pipe_ok):
        variant = 1
    if variant == 2:
        kernel_model.replay_gla_warp(bh, dk, dv, es, grid=None)
    elif variant == 3 or (variant == 0 and kernel_model.gla_auto_is_pipe(dk, dv, es)):
        kernel_model.replay_gla_pipe(bh, dk, dv, es)
    else:
        kernel_model.replay_gla(bh, dk, dv, es)
    gen = torch.Generator(device=cuda_dev)
    gen.manual_seed(case)
    q, k, v = ((torch.rand((bh, x), generator=gen, device=cuda_dev) * 2 - 1).to(dt) for x in (dk, dk, dv))
    gk = (-3 * torch.rand((bh, dk), generator=gen, device=cuda_dev)).to(dt)
    S = torch.randn((bh, dk, dv), generator=gen, device=cuda_dev).to(dt)
    S_in = S.clone()
    S_new, o = g.gla_decode(q, k, v, gk, S, scale=0.3, S_new=S if in_place else None, variant=variant)
    torch.cuda.synchronize()
    fmt = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}[dt]

    def bits(t):
        t = t.contiguous().cpu()
        return t.view(torch.int32).numpy().view(np.uint32) if dt == torch.float32 else \
            t.view(torch.int16).numpy().view(np.uint16)

    ref_S, ref_o, ss, os_ = oracle.gla_ref_decode(bits(q), bits(k), bits(v), bits(gk), bits(S_in), 0.3, fmt)
    u32 = 2.0 ** -24
    half_ulp = 0 if fmt == "f32" else 0.5
    tol_S = 8 * u32 * ss + half_ulp * parity_rules.ulp(ref_S, fmt)
    carried = 0.3 * np.einsum("hi,hij->hj", np.abs(q.double().cpu().numpy()), 8 * u32 * ss) if dk else 0.0
    tol_o = 1e-5 * os_ + carried + half_ulp * parity_rules.ulp(ref_o, fmt) + 1e-30
    label = f"gla case {case}: {bh}x{dk}x{dv} {fmt} variant {variant} in_place {in_place}"
    assert (np.abs(S_new.double().cpu().numpy() - ref_S) <= tol_S).all(), label
    assert (np.abs(o.double().cpu().numpy() - ref_o) <= tol_o).all(), label

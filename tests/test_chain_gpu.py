"""A decoder-layer chain on one stream: the GEMV projections of an input
vector feed one GLA decode step, whose output feeds the output projection,
for several tokens, with no synchronisation between the launches.

Every kernel here is a programmatic dependent launch, so each may start while
the one before it drains; this checks that every read of data the previous
kernel produces (a GEMV's input vector, the GLA step's q, k, v, gk and state,
the output projection's input) waits for it.  After one synchronisation at
the end, every stage of every token is checked against the oracle on the
values that stage actually read (the GEMV tolerances for the projections,
the GLA step's for the state and o).

Two launch modes:
  * defaults: gemv() and gla_decode() without configuration or flags;
  * promises: an ordinary copy starts every token (so nothing launched before
    it is still running), then the four input projections share their input
    under GEMV_OVERLAP_PDL_PREFETCH_BA (weights and input unwritten by the
    work in flight), the GLA step runs with GLA_PREFETCH_STATE (its state was
    written before that copy), and the output projection under
    GEMV_OVERLAP_PDL_PREFETCH_B (weights only: its input is the GLA output
    just produced).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import memory_bound_gemv_02_gb300 as g
import oracle
import parity_rules
from gpu_helpers import check_against_oracle

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


def _bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _check_gla(q, k, v, gk, S_in, S_new, o, scale, label):
    ref_S, ref_o, ss, os_ = oracle.gla_ref_decode(_bits(q), _bits(k), _bits(v), _bits(gk), _bits(S_in), scale, "bf16")
    got_S, got_o = S_new.double().cpu().numpy(), o.double().cpu().numpy()
    tol_S = 8 * U32 * ss + 0.5 * parity_rules.ulp(ref_S, "bf16")
    carried = abs(scale) * np.einsum("hi,hij->hj", np.abs(q.double().cpu().numpy()), 8 * U32 * ss)
    tol_o = 1e-5 * os_ + carried + 0.5 * parity_rules.ulp(ref_o, "bf16") + 1e-30
    assert (np.abs(got_S - ref_S) <= tol_S).all(), f"{label}: state"
    assert (np.abs(got_o - ref_o) <= tol_o).all(), f"{label}: o"


@pytest.mark.parametrize("mode", ["defaults", "promises"])
@pytest.mark.parametrize("H,D,DM", [(32, 64, 1024), (16, 128, 2048)])
def test_decoder_chain(cuda_dev, mode, H, D, DM):
    T, scale = 4, D ** -0.5
    gen = torch.Generator(device=cuda_dev)
    gen.manual_seed(H + D + DM)

    def w(rows, cols, sigma):
        return (torch.randn((rows, cols), generator=gen, device=cuda_dev) * sigma).to(torch.bfloat16)

    Wq, Wk, Wv = (w(H * D, DM, 0.05) for _ in range(3))
    Wg = w(H * D, DM, 0.02)
    Wo = w(DM, H * D, 0.05)
    xs = (torch.randn((T, DM), generator=gen, device=cuda_dev)).to(torch.bfloat16)
    states = [torch.randn((H, D, D), generator=gen, device=cuda_dev).to(torch.bfloat16)]
    states += [torch.empty_like(states[0]) for _ in range(T)]
    proj = {name: [torch.empty(H * D, dtype=torch.bfloat16, device=cuda_dev) for _ in range(T)]
            for name in ("q", "k", "v", "g")}
    outs = [torch.empty((H, D), dtype=torch.bfloat16, device=cuda_dev) for _ in range(T)]
    ys = [torch.empty(DM, dtype=torch.bfloat16, device=cuda_dev) for _ in range(T)]
    x_bufs = [torch.empty(DM, dtype=torch.bfloat16, device=cuda_dev) for _ in range(T)]
    torch.cuda.synchronize()

    shared = {"overlap": g.GEMV_OVERLAP_PDL_PREFETCH_BA}
    weights = {"overlap": g.GEMV_OVERLAP_PDL_PREFETCH_B}
    for t in range(T):
        if mode == "promises":
            x_bufs[t].copy_(xs[t])  # an ordinary operation: everything before it has completed
            x = x_bufs[t]
        else:
            x = xs[t]
        for name, W in (("q", Wq), ("k", Wk), ("v", Wv), ("g", Wg)):
            if mode == "promises":
                g.gemv_ex(W, x, c=proj[name][t], config=shared)
            else:
                g.gemv(W, x, c=proj[name][t])
        q, k, v, gk = (proj[n][t].view(H, D) for n in ("q", "k", "v", "g"))
        g.gla_decode(q, k, v, gk, states[t], scale, S_new=states[t + 1], o=outs[t],
                     flags=g.GLA_PREFETCH_STATE if mode == "promises" else 0)
        if mode == "promises":
            g.gemv_ex(Wo, outs[t].view(-1), c=ys[t], config=weights)
        else:
            g.gemv(Wo, outs[t].view(-1), c=ys[t])
    torch.cuda.synchronize()

    for t in range(T):
        label = f"{mode} token {t}"
        for name, W in (("q", Wq), ("k", Wk), ("v", Wv), ("g", Wg)):
            check_against_oracle(proj[name][t], W, xs[t], False, label=f"{label} {name}")
        q, k, v, gk = (proj[n][t].view(H, D) for n in ("q", "k", "v", "g"))
        _check_gla(q, k, v, gk, states[t], states[t + 1], outs[t], scale, label)
        check_against_oracle(ys[t], Wo, outs[t].view(-1), False, label=f"{label} y")

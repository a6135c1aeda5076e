"""The library's calls captured in a CUDA graph and replayed.

A sequence of every kernel family -- the tiles GEMV (default launch and the
shared-input promise), split-K with its second pass (workspace allocated
ahead with gemv_prepare on the capturing stream), the bulk kernel, the
fused epilogue, and the GLA step in its pipelined and CTA layouts -- is run
once eagerly on the capturing stream (plans, kernel attributes and the
workspace are set up then), captured into a torch.cuda.CUDAGraph (the
programmatic dependent launches become graph edges) and replayed on new
input values.  Each replay must equal the same sequence run eagerly, bit
for bit (same kernels, configurations and inputs), and its outputs are
checked against the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import memory_bound_gemv_02_gb300 as g
import oracle
import parity_rules
from gpu_helpers import check_against_oracle
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


def _bits16(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _same(x, y):
    v = (lambda t: t.view(torch.int32)) if x.dtype == torch.float32 else (lambda t: t.view(torch.int16))
    return torch.equal(v(x), v(y))


class Sequence:
    """Static buffers and the calls that read and write them."""

    def __init__(self, dev):
        self.dev = dev
        self.gen = torch.Generator(device=dev)
        bf, hf = torch.bfloat16, torch.float16
        self.B1 = torch.empty((3000, 4104), dtype=bf, device=dev)
        self.B1b = torch.empty((3000, 4104), dtype=bf, device=dev)
        self.a1 = torch.empty(4104, dtype=bf, device=dev)
        self.B2 = torch.empty((256, 262144), dtype=hf, device=dev)   # split-K
        self.a2 = torch.empty(262144, dtype=hf, device=dev)
        self.B3 = torch.empty((2048, 8195), dtype=hf, device=dev)    # bulk, unaligned rows
        self.a3 = torch.empty(8195, dtype=hf, device=dev)
        self.B4 = torch.empty((1000, 1000), dtype=bf, device=dev)    # fused epilogue
        self.a4 = torch.empty(1000, dtype=bf, device=dev)
        self.bias4 = torch.empty(1000, dtype=torch.float32, device=dev)
        H, D = 64, 64
        self.gla = [torch.empty(s, dtype=bf, device=dev) for s in ((H, D), (H, D), (H, D), (H, D), (H, D, D))]
        self.gla32 = [torch.empty(s, dtype=torch.float32, device=dev)
                      for s in ((32, 128), (32, 128), (32, 128), (32, 128), (32, 128, 128))]
        self.fill(0)

    def fill(self, seed):
        self.gen.manual_seed(seed)
        for t in (self.B1, self.B1b, self.a1, self.B2, self.a2, self.B3, self.a3, self.B4, self.a4):
            t.copy_(torch.rand(t.shape, generator=self.gen, device=self.dev) * 2 - 1)
        self.bias4.copy_(torch.rand(1000, generator=self.gen, device=self.dev) - 0.5)
        for lst in (self.gla, self.gla32):
            for i, t in enumerate(lst):
                x = torch.rand(t.shape, generator=self.gen, device=self.dev)
                t.copy_(-3 * x if i == 3 else 2 * x - 1)

    def outputs(self):
        dev, bf, hf = self.dev, torch.bfloat16, torch.float16
        return {"c1": torch.empty(3000, dtype=bf, device=dev), "c1b": torch.empty(3000, dtype=bf, device=dev),
                "c2": torch.empty(256, dtype=torch.float32, device=dev), "c3": torch.empty(2048, dtype=hf, device=dev),
                "c4": torch.empty(1000, dtype=torch.float32, device=dev),
                "S": torch.empty((64, 64, 64), dtype=bf, device=dev), "o": torch.empty((64, 64), dtype=bf, device=dev),
                "S32": torch.empty((32, 128, 128), dtype=torch.float32, device=dev),
                "o32": torch.empty((32, 128), dtype=torch.float32, device=dev)}

    def run(self, out):
        g.gemv(self.B1, self.a1, c=out["c1"])
        g.gemv_ex(self.B1b, self.a1, c=out["c1b"], config={"overlap": g.GEMV_OVERLAP_PDL_PREFETCH_BA})
        g.gemv(self.B2, self.a2, c=out["c2"], out_fp32=True)
        g.gemv_ex(self.B3, self.a3, c=out["c3"], config={"variant": g.GEMV_VARIANT_BULK, "overlap": 1})
        g.gemv_fused(self.B4, self.a4, c=out["c4"], out_fp32=True, alpha=0.5, beta=1.0, bias=self.bias4,
                     activation="silu")
        q, k, v, gk, S = self.gla
        g.gla_decode(q, k, v, gk, S, 0.125, S_new=out["S"], o=out["o"])
        q, k, v, gk, S = self.gla32
        g.gla_decode(q, k, v, gk, S, 0.1, S_new=out["S32"], o=out["o32"], variant=g.GLA_VARIANT_CTA)


def test_graph_capture_replay(cuda_dev):
    seq = Sequence(cuda_dev)
    s = torch.cuda.Stream(device=cuda_dev)
    graph_out = seq.outputs()
    eager_out = seq.outputs()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.gemv_prepare(256, 262144, g.GEMV_F16_OUT_F32, True, stream=s)
        seq.run(graph_out)  # eager warm-up on the capturing stream
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        seq.run(graph_out)
    torch.cuda.synchronize()

    for rep in range(3):
        seq.fill(100 + rep)
        graph.replay()
        seq.run(eager_out)
        torch.cuda.synchronize()
        for name in graph_out:
            assert _same(graph_out[name], eager_out[name]), f"replay {rep}: {name} differs from the eager run"
        check_against_oracle(graph_out["c1"], seq.B1, seq.a1, False, label=f"replay {rep} c1")
        check_against_oracle(graph_out["c1b"], seq.B1b, seq.a1, False, label=f"replay {rep} c1b")
        check_against_oracle(graph_out["c2"], seq.B2, seq.a2, True, label=f"replay {rep} split-K")
        check_against_oracle(graph_out["c3"], seq.B3, seq.a3, False, label=f"replay {rep} bulk")
        c_ref, s_ref = oracle.gemv_ref(inputs.to_bits(seq.B4), inputs.to_bits(seq.a4), "bf16")
        y_ref, scale = oracle.gemv_ref_epilogue(c_ref, s_ref, 0.5, 1.0, seq.bias4.cpu().numpy().view(np.uint32),
                                                "f32", "silu")
        got = graph_out["c4"].double().cpu().numpy()
        assert (np.abs(got - y_ref) <= 1e-5 * scale * 1.1 + 2e-6 * np.abs(y_ref) + 1e-30).all(), f"replay {rep} epilogue"
        q, k, v, gk, S = seq.gla
        ref_S, ref_o, ss, os_ = oracle.gla_ref_decode(*(_bits16(x) for x in (q, k, v, gk, S)), 0.125, "bf16")
        got_S = graph_out["S"].double().cpu().numpy()
        assert (np.abs(got_S - ref_S) <= 8 * U32 * ss + 0.5 * parity_rules.ulp(ref_S, "bf16")).all(), f"replay {rep} S"
        carried = 0.125 * np.einsum("hi,hij->hj", np.abs(q.double().cpu().numpy()), 8 * U32 * ss)
        tol_o = 1e-5 * os_ + carried + 0.5 * parity_rules.ulp(ref_o, "bf16") + 1e-30
        assert (np.abs(graph_out["o"].double().cpu().numpy() - ref_o) <= tol_o).all(), f"replay {rep} o"


def test_graph_replays_back_to_back(cuda_dev):
    """Ten replays of a graph of 16 GEMV calls on one input vector (the
    shared-input promise holds: nothing in the graph writes B or a), then
    the last outputs checked: replays may overlap only as the launches'
    programmatic edges allow."""
    dev = cuda_dev
    B, a = inputs.make_inputs(4096, 4096, "bf16", "uniform", 3, dev)
    Bs = [B] + [torch.roll(B, i, 0) for i in range(1, 4)]
    outs = [torch.empty(4096, dtype=torch.bfloat16, device=dev) for _ in range(16)]
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for i in range(16):
            g.gemv_ex(Bs[i % 4], a, c=outs[i], config={"overlap": g.GEMV_OVERLAP_PDL_PREFETCH_BA})
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for i in range(16):
            g.gemv_ex(Bs[i % 4], a, c=outs[i], config={"overlap": g.GEMV_OVERLAP_PDL_PREFETCH_BA})
    for _ in range(10):
        graph.replay()
    torch.cuda.synchronize()
    for i in range(4):
        check_against_oracle(outs[12 + i], Bs[i], a, False, label=f"graph output {12 + i}")
    for i in range(16):
        assert _same(outs[i], outs[i % 4])

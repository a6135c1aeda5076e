"""Concurrent use of the library from several host threads.

The header promises a thread-safe configuration cache and workspace table
and per-thread `gemv_last_config`.  Eight host threads, each on its own CUDA
stream, call gemv()/gemv_ex()/gla_decode() on a mix of shapes right after
the cache and workspaces were dropped (gemv_release), so they race to build
the same keys and to allocate their streams' split-K workspaces.  Every
result must be bit-identical to the same call made from one thread (same
shape and configuration give the same plan, hence the same summation
order), the references must match the oracle, and after each call a
thread's gemv_last_config must be the plan of its own call.
"""
from __future__ import annotations

import threading

import pytest
import torch

import memory_bound_gemv_02_gb300 as g
from gpu_helpers import check_against_oracle
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu

# (n, k, dtype, fp32 output, forced configuration)
CASES = [(1031, 4099, "f16", False, None), (300, 100003, "bf16", True, None),       # split-K planned
         (4096, 1000, "bf16", False, {"grid_split": 3}), (257, 7169, "f16", True, {"variant": 4}),
         (64, 16384, "f16", False, {"warp_split": 8}), (5000, 512, "bf16", True, None)]


def _call(B, a, out_fp32, cfg):
    return g.gemv_ex(B, a, out_fp32=out_fp32, config=cfg) if cfg else g.gemv(B, a, out_fp32=out_fp32)


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def test_eight_host_threads(cuda_dev):
    data = [inputs.make_inputs(n, k, dt, "uniform", 40 + i, cuda_dev) for i, (n, k, dt, _, _) in enumerate(CASES)]
    refs, plans = [], []
    for (n, k, dt, of, cfg), (B, a) in zip(CASES, data):
        c = _call(B, a, of, cfg)
        plans.append(g.gemv_last_config())
        torch.cuda.synchronize()
        check_against_oracle(c, B, a, of, label=f"reference {n}x{k}")
        refs.append(c)
    gq, gk_, gv, ggk, gS = (x.to(torch.bfloat16) for x in (torch.rand(64, 64, device=cuda_dev),
                                                            torch.rand(64, 64, device=cuda_dev),
                                                            torch.rand(64, 64, device=cuda_dev),
                                                            -torch.rand(64, 64, device=cuda_dev),
                                                            torch.randn(64, 64, 64, device=cuda_dev)))
    S_ref, o_ref = g.gla_decode(gq, gk_, gv, ggk, gS, scale=0.125)
    torch.cuda.synchronize()
    g.gemv_release()  # empty cache and workspaces: the threads race to rebuild them

    errors, results = [], [[] for _ in range(8)]

    def worker(tid):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for it in range(24):
                    i = (tid + it) % len(CASES)
                    n, k, dt, of, cfg = CASES[i]
                    B, a = data[i]
                    c = _call(B, a, of, cfg)
                    used = g.gemv_last_config()
                    if {kk: used[kk] for kk in plans[i]} != plans[i]:
                        errors.append(f"thread {tid}: last config {used} is not its own call's {plans[i]}")
                    results[tid].append((i, c))
                    if it % 6 == tid % 6:
                        results[tid].append(("gla", g.gla_decode(gq, gk_, gv, ggk, gS, scale=0.125)))
            s.synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append(f"thread {tid}: {e!r}")

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    torch.cuda.synchronize()
    assert not errors, errors[:4]
    for tid in range(8):
        assert len(results[tid]) >= 24
        for i, c in results[tid]:
            if i == "gla":
                S_new, o = c
                assert torch.equal(_bits(S_new), _bits(S_ref)) and torch.equal(_bits(o), _bits(o_ref)), tid
            else:
                assert torch.equal(_bits(c), _bits(refs[i])), (tid, CASES[i])

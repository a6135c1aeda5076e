"""The C-ABI boundary on a GPU: buffers outside the current device's memory
are refused with GEMV_ERR_DEVICE before anything is launched, and GEMV_LOG
prints one line per newly cached configuration.

Host buffers here are pinned (cudaMallocHost through torch), which the GPU
can address: even a broken check could not fault the device, it would only
compute into host memory -- which the tests would see.  Pageable host memory
is never passed."""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import pytest
import torch

import memory_bound_gemv_02_gb300 as g
from memory_bound_gemv_02_gb300 import inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _status(fn, *args):
    st = fn(*args)
    torch.cuda.synchronize()
    return st


def test_host_buffers_are_refused(cuda_dev):
    n, k = 96, 520
    B, a = inputs.make_inputs(n, k, "f16", "uniform", 3, cuda_dev)
    c = torch.full((n,), 5.0, dtype=torch.float16, device=cuda_dev)
    Bh, ah = B.cpu().pin_memory(), a.cpu().pin_memory()
    ch = torch.full((n,), 5.0, dtype=torch.float16).pin_memory()
    L = g.lib()
    s = torch.cuda.current_stream().cuda_stream
    for (Bx, ax, cx) in ((Bh, a, c), (B, ah, c), (B, a, ch)):
        st = _status(L.gemv, Bx.data_ptr(), ax.data_ptr(), cx.data_ptr(), n, k, g.GEMV_F16, s)
        assert st == g.GEMV_ERR_DEVICE
    assert (c == 5.0).all() and (ch == 5.0).all()  # nothing was written
    # the same through the other entry points that take device buffers
    cfg = g.GemvConfig()
    cfg.grid_split = 2
    assert _status(L.gemv_ex, Bh.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, 0, ctypes.byref(cfg),
                   s) == g.GEMV_ERR_DEVICE
    assert _status(L.gemv_splitk_noalloc, Bh.data_ptr(), a.data_ptr(), c.data_ptr(), n, k, 0, 2,
                   s) == g.GEMV_ERR_DEVICE
    ep = g.GemvEpilogue()
    ep.alpha, ep.beta, ep.bias_dtype = 1.0, 1.0, g.GEMV_BIAS_F32
    bias_h = torch.ones(n, dtype=torch.float32).pin_memory()
    ep.bias = bias_h.data_ptr()
    assert _status(L.gemv_fused, B.data_ptr(), k, a.data_ptr(), c.data_ptr(), n, k, 0, ctypes.byref(ep), None,
                   s) == g.GEMV_ERR_DEVICE
    # gemv_host: the device-side buffers must be device memory
    B_dev = torch.empty_like(B)
    assert _status(L.gemv_host, Bh.data_ptr(), ah.data_ptr(), ch.data_ptr(), Bh.data_ptr(), a.data_ptr(),
                   c.data_ptr(), n, k, 0, s) == g.GEMV_ERR_DEVICE
    assert (c == 5.0).all() and (ch == 5.0).all()
    # k == 0 writes only c: a host c is refused too
    assert _status(L.gemv, B.data_ptr(), a.data_ptr(), ch.data_ptr(), n, 0, 0, s) == g.GEMV_ERR_DEVICE
    assert (ch == 5.0).all()
    # and the valid call still works afterwards
    assert _status(L.gemv_host, Bh.data_ptr(), ah.data_ptr(), ch.data_ptr(), B_dev.data_ptr(), a.data_ptr(),
                   c.data_ptr(), n, k, 0, s) == g.GEMV_OK
    assert torch.equal(ch.to(cuda_dev), g.gemv(B, a))


def test_gla_host_state_is_refused(cuda_dev):
    bh, dk, dv = 4, 16, 64
    q, k, gk = (torch.zeros((bh, dk), dtype=torch.bfloat16, device=cuda_dev) for _ in range(3))
    v = torch.zeros((bh, dv), dtype=torch.bfloat16, device=cuda_dev)
    S_h = torch.ones((bh, dk, dv), dtype=torch.bfloat16).pin_memory()
    o = torch.full((bh, dv), 2.0, dtype=torch.bfloat16, device=cuda_dev)
    L = g.lib()
    st = _status(L.gla_decode, q.data_ptr(), k.data_ptr(), v.data_ptr(), gk.data_ptr(), S_h.data_ptr(),
                 S_h.data_ptr(), o.data_ptr(), bh, dk, dv, ctypes.c_float(1.0), g.GLA_BF16,
                 torch.cuda.current_stream().cuda_stream)
    assert st == g.GEMV_ERR_DEVICE
    assert (S_h == 1.0).all() and (o == 2.0).all()


CHILD = r"""
import sys
sys.path.insert(0, %r)
import torch
import memory_bound_gemv_02_gb300 as g
from memory_bound_gemv_02_gb300 import inputs
dev = torch.device("cuda", 0)
B, a = inputs.make_inputs(300, 1000, "bf16", "uniform", 0, dev)
B2, a2 = inputs.make_inputs(64, 4096, "f16", "uniform", 0, dev)
for _ in range(3):
    g.gemv(B, a)            # one new key, then cached
g.gemv(B, a, out_fp32=True)  # another key (fp32 output)
g.gemv_prepare(64, 4096, g.GEMV_F16, True)  # another, built ahead
g.gemv(B2, a2)              # already cached by gemv_prepare
g.gemv_ex(B, a, config={"warp_split": 2})  # forced: not cached, no line
torch.cuda.synchronize()
print("done")
""" % ROOT


def test_log_one_line_per_new_cached_config(cuda_dev):
    env = dict(os.environ, GEMV_LOG="1")
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("gemv:")]
    assert len(lines) == 3, lines
    assert lines[0].startswith("gemv: new config dev=0 n=300 k=1000 dtype=1 aligned=1 -> variant=")
    assert lines[1].startswith("gemv: new config dev=0 n=300 k=1000 dtype=3 aligned=1 -> variant=")
    assert lines[2].startswith("gemv: new config dev=0 n=64 k=4096 dtype=0 aligned=1 -> variant=")

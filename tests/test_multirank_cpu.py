"""The N>1 host paths on CPU with two gloo ranks: bench.py's max-over-ranks
timing reduction, and rows of one GEMV split across ranks (each rank owning
a contiguous block of rows of B and a replica of a), whose gathered result
must equal the single-process oracle exactly."""
from __future__ import annotations

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, _ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from memory_bound_gemv_02_gb300 import inputs
        m = bench.max_over_ranks(float(rank + 1) * 0.5, world)
        n, k = 37, 1003
        B, a = inputs.make_inputs(n, k, "bf16", "uniform", 4, "cpu")
        q, rem = divmod(n, world)
        r0 = rank * q + min(rank, rem)
        r1 = r0 + q + (1 if rank < rem else 0)
        c, _ = oracle.gemv_ref(inputs.to_bits(B[r0:r1]), inputs.to_bits(a), "bf16")
        parts = [None] * world
        dist.all_gather_object(parts, (r0, c.tolist()))
        if rank == 0:
            full = np.zeros(n)
            for s0, vals in parts:
                full[s0:s0 + len(vals)] = vals
            ref, _ = oracle.gemv_ref(inputs.to_bits(B), inputs.to_bits(a), "bf16")
            out.put((m, bool((full == ref).all())))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    m, same = q.get(timeout=10)
    assert m == 1.0 and same

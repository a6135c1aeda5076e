"""A host-side model of the streaming kernel's index arithmetic.

It replays, for a configuration from the planner, exactly the row, segment
and 16-byte-block ranges each CTA and warp of ``gemv_rows_kernel`` touches,
and the shared-memory, partial-sum and workspace indices it uses, so that the
following can be checked on the CPU before any launch:

* every element B[i, j] contributes exactly once (masked elements excluded);
* every global 16-byte block read lies inside the blocks that hold B;
* every shared-memory vector read lies inside the staged a segment, and the
  staged element read for (i, j) is a[j];
* cross-warp partial and split-K workspace indices stay in their buffers.
"""
from __future__ import annotations

import numpy as np


def _row_range(rbk, n, nrb):
    q, rem = divmod(n, nrb)
    r0 = rbk * q + min(rbk, rem)
    return r0, r0 + q + (1 if rbk < rem else 0)


def replay(n, k, cfg, base_off=0, ldb=None):
    """Return a dict of findings; raises AssertionError on any violation.
    ``ldb``: row stride of B in elements (default k)."""
    ldb = k if ldb is None else ldb
    if cfg["variant"] == 3:
        return replay_tiles(n, k, cfg, base_off, ldb)
    if cfg["variant"] == 4:
        return replay_bulk(n, k, cfg, base_off, ldb)
    assert ldb == k, "row-per-warp replay models ldb == k only"
    W, R, Sw, Sg = cfg["warps_per_cta"], cfg["rows_per_warp"], cfg["warp_split"], cfg["grid_split"]
    nrb, kseg, variant, ctas = cfg["row_blocks"], cfg["k_segment"], cfg["variant"], cfg["ctas"]
    assert ctas == nrb * Sg and W % Sw == 0
    as_elems = -(-(kseg + 24) // 8) * 8
    assert cfg["smem_bytes"] == as_elems * 2 + W * R * 4
    cover = np.zeros((n, k), dtype=np.int32)
    total_elems = base_off + n * k  # elements from the aligned base
    nblocks = -(-total_elems // 8)  # 16-byte blocks that hold any byte of B
    ws_rows = set()
    slots = W // Sw
    for cta in range(ctas):
        gs, rbk = cta % Sg, cta // Sg
        r0, r1 = _row_range(rbk, n, nrb)
        j0 = gs * kseg
        seglen = min(k - j0, kseg)
        assert seglen >= 1, "empty k-segment"
        if Sg > 1:
            assert j0 % 8 == 0
        for base in range(r0, r1, slots * R):
            for warp in range(W):
                slot, s = divmod(warp, Sw)
                i0 = base + slot * R
                if Sw > 1:
                    for r in range(R):
                        assert 0 <= (slot * R + r) * Sw + s < W * R
                if variant == 1:
                    assert base_off == 0 and k % 8 == 0 and seglen % 8 == 0
                    nt = seglen // 8
                    t0, t1 = nt * s // Sw, nt * (s + 1) // Sw
                    if t1 <= t0:
                        continue
                    t = np.arange(t0, t1)
                    assert ((t + 1) * 8 + 7 < as_elems).all()
                    for r in range(R):
                        row = i0 + r if i0 + r < r1 else i0  # rows past r1 re-read row i0
                        if i0 >= r1:
                            break
                        blk = (row * k + j0) // 8 + t
                        assert blk.min() >= 0 and blk.max() < nblocks
                        if i0 + r < r1:
                            cols = (j0 + 8 * t[:, None] + np.arange(8)[None, :]).ravel()
                            np.add.at(cover[row], cols, 1)
                else:
                    assert R == 1
                    if i0 >= r1:
                        continue
                    e0 = base_off + i0 * k + j0
                    g0, off = e0 >> 3, e0 & 7
                    nt = (off + seglen + 7) >> 3
                    t0, t1 = nt * s // Sw, nt * (s + 1) // Sw
                    if t1 <= t0:
                        continue
                    last_hi = seglen + off - 8 * (nt - 1)
                    assert 1 <= last_hi <= 8
                    t = np.arange(t0, t1)
                    blk = g0 + t
                    assert blk.min() >= 0 and blk.max() < nblocks
                    assert ((t + 1) * 8 + 7 < as_elems).all()  # as4[t + 1] (and as4[t]) in range
                    p = np.arange(8)[None, :]
                    tt = t[:, None]
                    valid = ((tt > 0) | (p >= off)) & ((tt < nt - 1) | (p < last_hi))
                    # staged index of element p of block t, and the column it holds
                    x = 8 * tt + (8 - off) + p
                    col_from_stage = j0 + x - 8
                    elem = 8 * blk[:, None] + p - base_off  # flat element index in B
                    col_from_B = elem - i0 * k
                    assert (col_from_stage[valid] == col_from_B[valid]).all()
                    assert (x[valid] >= 8).all() and (x[valid] < 8 + seglen).all()
                    np.add.at(cover[i0], col_from_B[valid], 1)
        if Sg > 1:
            for row in range(r0, r1):
                idx = gs * n + row
                assert 0 <= idx < Sg * n
                ws_rows.add(idx)
    assert (cover == 1).all(), f"coverage wrong: min {cover.min()} max {cover.max()}"
    if Sg > 1:
        assert len(ws_rows) == Sg * n
    return {"ctas": ctas}


def replay_tiles(n, k, cfg, base_off=0, ldb=None):
    """The same checks for ``gemv_tiles_kernel`` (row i of B starts at
    element i * ldb)."""
    ldb = k if ldb is None else ldb
    W, R, S, Sg = cfg["warps_per_cta"], cfg["rows_per_warp"], cfg["warp_split"], cfg["grid_split"]
    C, kseg, U, ctas = cfg["row_blocks"], cfg["k_segment"], cfg["unroll"], cfg["ctas"]
    aligned = base_off == 0 and k % 8 == 0 and ldb % 8 == 0
    NCLS = 1 if aligned else 8
    assert ctas == C * Sg and W % S == 0 and C % NCLS == 0 and C >= NCLS
    assert (R, U) in ((1, 8), (1, 4), (2, 4), (4, 2))
    as_elems = -(-(kseg + 24) // 8) * 8
    assert cfg["smem_bytes"] == as_elems * 2 + 2 * W * R * 4
    slots = W // S
    if S > 1:
        assert 1 + slots - 1 <= 15  # named barrier ids 1..slots
    cover = np.zeros((n, k), dtype=np.int32)
    nblocks = -(-(base_off + (n - 1) * ldb + k) // 8)  # blocks holding any byte of B's rows
    ws_rows = set()
    Cq = C // NCLS
    for cta in range(ctas):
        gs, c = cta % Sg, cta // Sg
        cls, cq = c % NCLS, c // NCLS
        j0 = gs * kseg
        seglen = min(k - j0, kseg)
        assert seglen >= 1
        nr = (n - cls + NCLS - 1) // NCLS if n > cls else 0
        off = 0 if aligned else (base_off + j0 + cls * (ldb & 7)) & 7
        nt = (off + seglen + 7) >> 3
        last_hi = seglen + off - 8 * (nt - 1)
        assert 1 <= last_hi <= 8
        assert nt <= as_elems // 8
        RT = slots * R
        L = -(-nt // S)
        nloc = -(-(nr - cq) // Cq) if nr > cq else 0
        ngroups = -(-nloc // RT)
        stage_x = np.arange(8 * nt)
        stage_col = stage_x - off  # segment column held by staged element x
        if ngroups > 0:
            # L2 prefetch of the second step, issued with B promised unwritten:
            # the next 32*U blocks of the first tile's row slices.  Every
            # prefetched block must be a block of that row's own slice.
            for warp in range(W):
                slot, s = divmod(warp, S)
                t0 = min(s * L, nt)
                t1 = min(t0 + L, nt)
                b0 = t0 + 32 * U
                b1 = min(b0 + 32 * U, t1)
                for r in range(R):
                    m = slot * R + r
                    if m >= nloc or b1 <= b0:
                        continue
                    i = NCLS * (cq + Cq * m) + cls
                    g0 = (base_off + i * ldb + j0) >> 3
                    assert t0 <= b0 < b1 <= t1 and b1 - b0 <= 32 * U
                    assert 0 <= g0 + b0 and g0 + b1 <= nblocks
        for g in range(ngroups):
            for warp in range(W):
                slot, s = divmod(warp, S)
                mb = g * RT + slot * R
                t0 = min(s * L, nt)
                t1 = min(t0 + L, nt)
                if S > 1:
                    for r in range(R):
                        assert 0 <= (slot * R + r) * S + s < W * R
                for r in range(R):
                    m = mb + r
                    if m >= nloc:
                        continue
                    j = cq + Cq * m
                    assert j < nr
                    i = NCLS * j + cls
                    assert i < n
                    e0 = base_off + i * ldb + j0
                    assert (e0 & 7) == off, "row offset differs inside a CTA"
                    g0 = e0 >> 3
                    if t1 <= t0:
                        continue
                    t = np.arange(t0, t1)
                    blk = g0 + t
                    assert blk.min() >= 0 and blk.max() < nblocks
                    p = np.arange(8)[None, :]
                    tt = t[:, None]
                    if aligned:
                        valid = np.ones((t.size, 8), bool)
                    else:
                        valid = ((tt > 0) | (p >= off)) & ((tt < nt - 1) | (p < last_hi))
                    elem = 8 * blk[:, None] + p - base_off
                    col_B = elem - i * ldb - j0
                    col_stage = stage_col[8 * tt + p]
                    assert (col_B[valid] == col_stage[valid]).all()
                    assert (col_B[valid] >= 0).all() and (col_B[valid] < seglen).all()
                    # outside the row the staged a must be zero (the kernel relies on it)
                    outside = ~valid
                    assert ((col_stage[outside] < 0) | (col_stage[outside] >= seglen)).all()
                    np.add.at(cover[i], j0 + col_B[valid], 1)
                    if Sg > 1:
                        ws_rows.add(gs * n + i)
    assert (cover == 1).all(), f"coverage wrong: min {cover.min()} max {cover.max()}"
    if Sg > 1:
        assert len(ws_rows) == Sg * n
    return {"ctas": ctas}


def replay_bulk(n, k, cfg, base_off=0, ldb=None):
    """The same checks for ``gemv_bulk_kernel``, plus its ring: lane 0's
    issue cursor and the warp's consume cursor are replayed side by side, so
    that every bulk copy is checked (source blocks inside B, 16-byte aligned,
    size a multiple of 16 and at most one buffer; destination inside the
    warp's own ring; mbarrier inside shared memory), every buffer is refilled
    only after it was consumed, every wait uses the parity of the phase that
    the chunk it expects completes, and the consumed chunks cover each row
    slice exactly once."""
    ldb = k if ldb is None else ldb
    W, R, S, Sg = cfg["warps_per_cta"], cfg["rows_per_warp"], cfg["warp_split"], cfg["grid_split"]
    C, kseg, U, ctas, NS = cfg["row_blocks"], cfg["k_segment"], cfg["unroll"], cfg["ctas"], cfg["stages"]
    aligned = base_off == 0 and k % 8 == 0 and ldb % 8 == 0
    NCLS = 1 if aligned else 8
    assert R == 1 and U in (4, 8) and 2 <= NS <= 8
    assert ctas == C * Sg and W % S == 0 and C % NCLS == 0 and C >= NCLS
    SB = 32 * U
    as_elems = -(-(kseg + 24) // 8) * 8
    ring_off = -(-(as_elems * 2 + 8 * W) // 128) * 128
    ring_bytes = W * NS * SB * 16
    smem = cfg["smem_bytes"]
    assert smem == ring_off + W * NS * (512 * U + 8) and smem <= 232448
    assert as_elems * 2 + 2 * W * 4 <= ring_off  # a and the partials end before the rings
    slots = W // S
    if S > 1:
        assert slots <= 15  # named barrier ids 1..slots
    cover = np.zeros((n, k), dtype=np.uint8)  # 0 or 1 expected; uint8 keeps full-size replays small
    nblocks = -(-(base_off + (n - 1) * ldb + k) // 8)
    Cq = C // NCLS
    ws_rows = set()
    for cta in range(ctas):
        gs, c = cta % Sg, cta // Sg
        cls, cq = c % NCLS, c // NCLS
        j0 = gs * kseg
        seglen = min(k - j0, kseg)
        assert seglen >= 1
        nr = (n - cls + NCLS - 1) // NCLS if n > cls else 0
        off = 0 if aligned else (base_off + j0 + cls * (ldb & 7)) & 7
        nt = (off + seglen + 7) >> 3
        last_hi = seglen + off - 8 * (nt - 1)
        assert 1 <= last_hi <= 8 and nt <= as_elems // 8
        RT = slots
        L = -(-nt // S)
        nloc = -(-(nr - cq) // Cq) if nr > cq else 0
        ngroups = -(-nloc // RT)
        stage_col = np.arange(8 * nt) - off

        def row_of(m):
            return NCLS * (cq + Cq * m) + cls

        for warp in range(W):
            slot, s = divmod(warp, S)
            t0 = min(s * L, nt)
            t1 = min(t0 + L, nt)
            nst = -(-(t1 - t0) // SB)
            gv = -(-(nloc - slot) // RT) if nloc > slot else 0
            total = gv * nst
            bufs = [None] * NS      # chunk held (or in flight) per buffer
            phases = [0] * NS       # phases completed per buffer once its copy lands
            cur = {"ic": 0, "ig": 0, "ist": 0, "ib": 0}

            def issue():
                ib, ig, ist = cur["ib"], cur["ig"], cur["ist"]
                assert bufs[ib] is None, "buffer refilled before it was consumed"
                tb = t0 + ist * SB
                nb = min(SB, t1 - tb)
                assert 1 <= nb <= SB
                i = row_of(ig * RT + slot)
                e0 = base_off + i * ldb + j0
                assert (e0 & 7) == off
                src = (e0 >> 3) + tb
                assert 0 <= src and src + nb <= nblocks
                dst = ring_off + (warp * NS + ib) * SB * 16
                assert dst % 16 == 0 and dst + nb * 16 <= ring_off + ring_bytes
                assert ring_off + (warp * NS + ib) * SB * 16 + SB * 16 <= ring_off + ring_bytes
                bar = ring_off + ring_bytes + (warp * NS + ib) * 8
                assert bar % 8 == 0 and bar + 8 <= smem
                bufs[ib] = (cur["ic"], ig, ist, src, nb)
                cur["ic"] += 1
                cur["ib"] = (ib + 1) % NS
                cur["ist"] += 1
                if cur["ist"] == nst:
                    cur["ist"] = 0
                    cur["ig"] += 1

            while cur["ic"] < total and cur["ic"] < NS:
                issue()
            cb, cpar, consumed = 0, 0, 0
            for g in range(ngroups):
                if g >= gv:
                    continue
                i = row_of(g * RT + slot)
                assert i < n
                for st in range(nst):
                    held = bufs[cb]
                    assert held is not None and held[1] == g and held[2] == st, "buffer holds the wrong chunk"
                    cidx, _, _, src, nb = held
                    assert cidx == consumed
                    # the wait on parity cpar completes with this chunk's phase
                    assert (phases[cb] & 1) == cpar
                    phases[cb] += 1
                    tb = t0 + st * SB
                    assert nb == min(SB, t1 - tb)
                    t = np.arange(tb, tb + nb)
                    blk = src + np.arange(nb)
                    p = np.arange(8)[None, :]
                    tt = t[:, None]
                    if aligned:
                        valid = np.ones((t.size, 8), bool)
                    else:
                        valid = ((tt > 0) | (p >= off)) & ((tt < nt - 1) | (p < last_hi))
                    elem = 8 * blk[:, None] + p - base_off
                    col_B = elem - i * ldb - j0
                    col_stage = stage_col[8 * tt + p]
                    assert (col_B[valid] == col_stage[valid]).all()
                    assert ((col_stage[~valid] < 0) | (col_stage[~valid] >= seglen)).all()
                    np.add.at(cover[i], j0 + col_B[valid], 1)
                    bufs[cb] = None
                    consumed += 1
                    if cur["ic"] < total:
                        assert cur["ib"] == cb  # the refill goes into the buffer just consumed
                        issue()
                    cb += 1
                    if cb == NS:
                        cb, cpar = 0, cpar ^ 1
                if Sg > 1:
                    ws_rows.add(gs * n + i)
            assert cur["ic"] == total == consumed
    assert (cover == 1).all(), f"coverage wrong: min {cover.min()} max {cover.max()}"
    if Sg > 1:
        assert len(ws_rows) == Sg * n
    return {"ctas": ctas}


def staged_shifted(a, j0, seglen, off, as_elems):
    """Host model of the tiles kernel's staging: output vector q is elements
    [8 - off, 16 - off) of source vectors (q - 1) ++ q, source vector q being
    a[j0 + 8q .. j0 + 8q + 7] with zeros outside the segment."""
    def src(q):
        v = np.zeros(8, dtype=a.dtype)
        for e in range(8):
            j = 8 * q + e
            if q >= 0 and 0 <= j < seglen:
                v[e] = a[j0 + j]
        return v
    out = np.zeros(as_elems, dtype=a.dtype)
    sh = 8 - off
    for q in range(as_elems // 8):
        pair = np.concatenate([src(q - 1), src(q)])
        out[8 * q: 8 * q + 8] = pair[sh: sh + 8]
    return out



def staging_schedule(nvec, block, shifted):
    """Replay of the staging loop's thread schedule (``stage_shift_loop``):
    unshifted, thread x of a ``block``-thread CTA first takes pairs
    (q, q + block) for q = x, x + 2*block, ... while q + block < ``nvec``
    (both loads before either store), then single vectors; shifted, single
    vectors only.  Checks that every output vector is written exactly once
    and every load address is inside [0, nvec).  Returns the largest number
    of paired iterations of a thread."""
    writes = np.zeros(nvec, dtype=np.int64)
    most = 0
    for x in range(block):
        q = x
        it = 0
        if not shifted:
            while q + block < nvec:
                assert 0 <= q and q + block < nvec
                writes[q] += 1
                writes[q + block] += 1
                q += 2 * block
                it += 1
        while q < nvec:
            writes[q] += 1
            q += block
        most = max(most, it)
    assert (writes == 1).all(), f"vectors written {writes.min()}..{writes.max()} times"
    return most


def gla_partial_store_conflicts(cpr, vec, dv):
    """Bank-conflict count of the GLA partial stores (``store_partials``):
    a warp's lanes (column chunk cc = lane % cpr, row block lane // cpr) each
    store VEC floats at float offset (row block * dv + cc * vec) as 16-byte
    vectors -- for VEC = 8 the half (bit 5 of the offset) first.  Each store
    instruction is served in phases of 8 lanes; a phase conflicts where two
    lanes hit the same 16-byte bank group (offset / 4 mod 8).  Returns the
    number of extra wavefronts over the warp's stores."""
    extra = 0
    halves = vec // 4
    for step in range(halves):
        for phase in range(4):
            groups = []
            for lane in range(8 * phase, 8 * phase + 8):
                cc, rb = lane % cpr, lane // cpr
                base = rb * dv + cc * vec
                h = step if vec == 4 else (step ^ ((base >> 5) & 1))
                off = base + 4 * h
                assert off % 4 == 0
                groups.append((off // 4) % 8)
            extra += max(groups.count(gr) for gr in set(groups)) - 1
    return extra


def gla_store_o_schedule(nh, G, dv, RP, nthreads=256):
    """Replay of the GLA step's o epilogue (``store_o``, four outputs per
    thread): thread t takes outputs x = 4 * x4 .. 4 * x4 + 3 for x4 = t,
    t + nthreads, ... < nh * dv / 4, reading the 16-byte partials at float
    offset (g * RP + rb) * dv + j (x = g * dv + j) for rb < RP.  Checks that
    every output of the round is written once, that the four outputs of a
    thread belong to one head (j % 4 == 0, dv % 4 == 0), and that every
    partial read is 16-byte aligned and inside part[G][RP][dv]."""
    assert dv % 4 == 0 and nh <= G
    writes = np.zeros(nh * dv, dtype=np.int64)
    for t in range(nthreads):
        for x4 in range(t, nh * dv // 4, nthreads):
            x = 4 * x4
            g, j = divmod(x, dv)
            assert j + 3 < dv and g < nh
            for rb in range(RP):
                off = (g * RP + rb) * dv + j
                assert off % 4 == 0 and 0 <= off and off + 4 <= G * RP * dv
            writes[x:x + 4] += 1
    assert (writes == 1).all()


def gla_balanced_grid(units, cap):
    """The host's grid for `units` rounds dealt round-robin over at most
    `cap` resident CTAs: the fewest rounds per CTA, then the fewest CTAs --
    unless that is below 4/5 of the cap, which then stays."""
    if units <= cap:
        return units
    per = -(-units // cap)
    grid = -(-units // per)
    return grid if 5 * grid >= 4 * cap else cap


def gla_rows_in_flight(dk, cpr):
    """The host's choice of rows in flight per thread: 8 for heads of at most
    1024 16-byte chunks, else 4."""
    return 8 if dk * cpr <= 1024 else 4


def gla_heads_per_cta(bh, dk, cpr, threads=256, rows_in_flight=None):
    """The host's choice of heads processed side by side per CTA round."""
    if rows_in_flight is None:
        rows_in_flight = gla_rows_in_flight(dk, cpr)
    G = 1
    while 2 * G * cpr <= threads and 2 * G <= bh and dk * cpr * 2 * G <= rows_in_flight * threads:
        G *= 2
    return G


def replay_gla(bh, dk, dv, elem_bytes, threads=256, rows_in_flight=None, grid=None):
    """Index replay of ``gla_decode_kernel`` (G heads per CTA round): every
    state element of every head is read and written exactly once by one
    thread, every staging, partial and output index is in range, and every
    partial read by the o reduction was written in the same round."""
    vec = 16 // elem_bytes
    assert dv % vec == 0
    cpr = dv // vec
    assert 1 <= cpr <= threads
    if rows_in_flight is None:
        rows_in_flight = gla_rows_in_flight(dk, cpr)
    G = gla_heads_per_cta(bh, dk, cpr, threads, rows_in_flight)
    assert G * cpr <= threads and threads % G == 0
    TPG = threads // G
    RP = TPG // cpr
    assert RP >= 1
    P0 = 3 * G * dk + (-(3 * G * dk)) % 4  # partials start on a 16-byte boundary
    smem_floats = P0 + G * RP * dv
    rounds = -(-bh // G)
    grid = rounds if grid is None else min(grid, rounds)
    touched = np.zeros((bh, dk, dv), dtype=np.int32)
    o_written = np.zeros((bh, dv), dtype=np.int32)
    for blk in range(grid):
        for r in range(blk, rounds, grid):
            h0 = r * G
            nh = min(G, bh - h0)
            part_written = set()
            for t in range(threads):
                gi, tl = divmod(t, TPG)
                cc, rl = tl % cpr, tl // cpr
                if not (rl < RP and gi < nh):
                    continue
                h = h0 + gi
                for i0 in range(rl, dk, RP * rows_in_flight):
                    for u in range(rows_in_flight):
                        i = i0 + u * RP
                        if i < dk:
                            vidx = (h * dk + i) * cpr + cc
                            assert 0 <= vidx < bh * dk * cpr
                            assert 2 * G * dk + gi * dk + i < 3 * G * dk  # qq[gi][i], the last staged array
                            touched[h, i, cc * vec:(cc + 1) * vec] += 1
                base = P0 + (gi * RP + rl) * dv + cc * vec
                assert base + vec <= smem_floats and base % 4 == 0  # 16-byte vector stores
                part_written.update(range(base, base + vec))
                assert (h * dv) // vec + cc < bh * dv // vec
            for x in range(nh * dv):
                g, j = divmod(x, dv)
                for rb in range(RP):
                    assert P0 + (g * RP + rb) * dv + j in part_written
                o_written[h0 + g, j] += 1
    assert (touched == 1).all() and (o_written == 1).all()
    return {"smem_floats": smem_floats, "heads_per_cta": G}


GLA_PIPE_ROUND_CHUNKS = 2048


GLA_PIPE_MAX_SMEM = 110 * 1024


def gla_pipe_smem(G, dk, dv, elem_bytes, threads=256):
    cpr = dv * elem_bytes // 16
    RP = threads // G // cpr
    return 2 * 16 * (G * dk * cpr + 3 * (G * dk * elem_bytes // 16) + G * cpr) + 4 * G * RP * dv + 3 * 4 * G * dk


def gla_pipe_ok(dk, dv, elem_bytes):
    """The host's condition for the pipelined layout (aligned pointers
    assumed): q, k, gk rows of whole 16-byte chunks, one head within a round
    and its buffers within the shared-memory budget."""
    cpr = dv * elem_bytes // 16
    return (dk > 0 and (dk * elem_bytes) % 16 == 0 and dk * cpr <= GLA_PIPE_ROUND_CHUNKS
            and gla_pipe_smem(1, dk, dv, elem_bytes) <= GLA_PIPE_MAX_SMEM)


def gla_auto_is_pipe(dk, dv, elem_bytes):
    """The automatic choice (aligned pointers assumed): the pipelined layout
    where it applies, else the CTA layout."""
    return gla_pipe_ok(dk, dv, elem_bytes)


def gla_pipe_heads_per_cta(bh, dk, dv, elem_bytes, threads=256):
    cpr = dv * elem_bytes // 16
    G = 1
    while (2 * G * cpr <= threads and 2 * G <= bh and dk * cpr * 2 * G <= GLA_PIPE_ROUND_CHUNKS
           and gla_pipe_smem(2 * G, dk, dv, elem_bytes, threads) <= GLA_PIPE_MAX_SMEM):
        G *= 2
    return G


def replay_gla_pipe(bh, dk, dv, elem_bytes, threads=256, grid=None):
    """Index replay of ``gla_decode_pipe_kernel``: per CTA, round r's copies
    go to buffer j % 2 (j = the CTA's round count so far) -- every state
    chunk copied once, by the thread that later reads it, from inside S into
    inside its buffer; q, k, gk, v chunks copied once per round from inside
    their arrays; every staged element read by the compute was copied for
    that round into that buffer; no copy targets the buffer a round still
    reads; partials and o as in the CTA layout; the shared-memory size is
    the host's."""
    vec = 16 // elem_bytes
    cpr = dv // vec
    assert gla_pipe_ok(dk, dv, elem_bytes) and 1 <= cpr <= threads
    G = gla_pipe_heads_per_cta(bh, dk, dv, elem_bytes, threads)
    TPG = threads // G
    RP = TPG // cpr
    assert RP >= 1 and G * dk * cpr <= GLA_PIPE_ROUND_CHUNKS
    SC, QC = G * dk * cpr, G * dk * elem_bytes // 16
    BUF = SC + 3 * QC + G * cpr
    PARTS = 2 * BUF * 16                    # byte offset of o's partials
    FACT = PARTS + G * RP * dv * 4          # byte offset of the fp32 exp(gk), k, q
    smem = FACT + 3 * G * dk * 4
    assert smem == gla_pipe_smem(G, dk, dv, elem_bytes, threads) <= GLA_PIPE_MAX_SMEM
    rounds = -(-bh // G)
    grid = rounds if grid is None else min(grid, rounds)
    s_chunks, q_chunks, v_chunks = bh * dk * cpr, bh * dk * elem_bytes // 16, bh * cpr
    read = np.zeros(s_chunks, dtype=np.int32)
    vec_copied = np.zeros((3, q_chunks), dtype=np.int32)
    v_copied = np.zeros(v_chunks, dtype=np.int32)
    o_written = np.zeros((bh, dv), dtype=np.int32)

    def copies(r, b):
        """{(smem chunk): (kind, global chunk, thread)} of round r into buffer b."""
        out = {}
        h0 = r * G
        nh = min(G, bh - h0)
        for t in range(threads):
            gi, tl = divmod(t, TPG)
            cc, rl = tl % cpr, tl // cpr
            if rl < RP and gi < nh:
                for i in range(rl, dk, RP):
                    dst = b * BUF + (gi * dk + i) * cpr + cc
                    src = ((h0 + gi) * dk + i) * cpr + cc
                    assert dst not in out and 0 <= src < s_chunks
                    out[dst] = ("S", src, t)
        nq, nv = nh * dk * elem_bytes // 16, nh * cpr
        q0 = h0 * dk * elem_bytes // 16
        for t in range(threads):
            for x in range(t, 3 * nq + nv, threads):
                if x < 3 * nq:
                    a, y = divmod(x, nq)
                    dst, src = b * BUF + SC + a * QC + y, q0 + y
                    assert 0 <= src < q_chunks and y < QC
                    out[dst] = ("qkg"[a], src, t)
                else:
                    y = x - 3 * nq
                    dst, src = b * BUF + SC + 3 * QC + y, h0 * cpr + y
                    assert 0 <= src < v_chunks and y < G * cpr
                    out[dst] = ("v", src, t)
        for dst in out:
            assert b * BUF <= dst < (b + 1) * BUF
        return out

    for blk in range(grid):
        my = list(range(blk, rounds, grid))
        pending = {0: copies(my[0], 0)} if my else {}
        for j, r in enumerate(my):
            b = j % 2
            if j + 1 < len(my):
                nxt = copies(my[j + 1], b ^ 1)
                assert all(d // BUF == b ^ 1 for d in nxt)  # never the buffer round j reads
                pending[b ^ 1] = nxt
            cur = pending.pop(b)
            for kind, src, _ in cur.values():
                if kind in "qkg":
                    vec_copied["qkg".index(kind), src] += 1
                elif kind == "v":
                    v_copied[src] += 1
            h0 = r * G
            nh = min(G, bh - h0)
            # the fp32 factors: element x of exp(gk), k and q (x < nh * dk,
            # written by thread x % threads) from the buffer's q, k, gk chunks
            converted = set()
            for t in range(threads):
                for x in range(t, nh * dk, threads):
                    for a in range(3):
                        qsm = b * BUF + SC + a * QC + (x * elem_bytes) // 16
                        assert cur[qsm][0] == "qkg"[a]
                        off = FACT + 4 * (a * G * dk + x)
                        assert FACT <= off and off + 4 <= smem
                    converted.add(x)
            for t in range(threads):
                gi, tl = divmod(t, TPG)
                cc, rl = tl % cpr, tl // cpr
                if not (rl < RP and gi < nh):
                    continue
                h = h0 + gi
                vsm = b * BUF + SC + 3 * QC + gi * cpr + cc
                assert cur[vsm][0] == "v" and cur[vsm][1] == h * cpr + cc
                for i in range(rl, dk, RP):
                    sm = b * BUF + (gi * dk + i) * cpr + cc
                    kind, src, owner = cur[sm]
                    assert kind == "S" and owner == t and src == (h * dk + i) * cpr + cc
                    read[src] += 1
                    x = gi * dk + i  # element of q, k, gk in the buffer and of the fp32 factors
                    assert x in converted
                    for a in range(3):
                        qsm = b * BUF + SC + a * QC + (x * elem_bytes) // 16
                        assert cur[qsm][0] == "qkg"[a]
                        assert cur[qsm][1] * 16 // elem_bytes + (x * elem_bytes % 16) // elem_bytes == h * dk + i
                base = PARTS + ((gi * RP + rl) * dv + cc * vec) * 4
                assert base + 4 * vec <= FACT and base % 16 == 0
            for x in range(nh * dv):
                g, jj = divmod(x, dv)
                o_written[h0 + g, jj] += 1
    assert (read == 1).all() and (o_written == 1).all()
    assert (vec_copied == 1).all() and (v_copied == 1).all()
    return {"smem_bytes": smem, "heads_per_cta": G}


def replay_gla_warp(bh, dk, dv, elem_bytes, warps_per_cta=8, grid=None, rows_in_flight=8):
    """Index replay of ``gla_decode_warp_kernel``: warp w of the grid takes
    heads w, w + warps, ...; lane l owns chunk l % cpr of rows l // cpr +
    RPW * m.  Every state element of every head is read and written exactly
    once, every shuffle source lane is a lane of the warp holding the same
    chunk, and every o chunk is stored once."""
    vec = 16 // elem_bytes
    assert dv % vec == 0
    cpr = dv // vec
    assert 1 <= cpr <= 32
    RPW = 32 // cpr
    heads_per_grid = None
    nwarps_total = -(-bh // warps_per_cta) * warps_per_cta
    if grid is not None:
        nwarps_total = min(grid, -(-bh // warps_per_cta)) * warps_per_cta
    heads_per_grid = nwarps_total
    touched = np.zeros((bh, dk, dv), dtype=np.int32)
    o_written = np.zeros((bh, dv), dtype=np.int32)
    for w in range(nwarps_total):
        for h in range(w, bh, heads_per_grid):
            for lane in range(32):
                cc, rw = lane % cpr, lane // cpr
                if rw < RPW:
                    for i0 in range(rw, dk, RPW * rows_in_flight):
                        for u in range(rows_in_flight):
                            i = i0 + u * RPW
                            if i < dk:
                                vidx = (h * dk + i) * cpr + cc
                                assert 0 <= vidx < bh * dk * cpr
                                touched[h, i, cc * vec:(cc + 1) * vec] += 1
                # the o reduction reads lanes cc + r * cpr, r < RPW: same chunk, every row group
                srcs = [cc + r * cpr for r in range(RPW)]
                assert all(0 <= x < 32 and x % cpr == cc for x in srcs)
                assert sorted(x // cpr for x in srcs) == list(range(RPW))
                if rw == 0:
                    assert 0 <= h * cpr + cc < bh * cpr
                    o_written[h, cc * vec:(cc + 1) * vec] += 1
    assert (touched == 1).all() and (o_written == 1).all()
    return {"warps": nwarps_total}

// "Tiles" GEMV kernel for sm_103a: c = B @ a, B (n, k) row-major, fp16/bf16
// in, fp32 accumulation (TileLang Case Studies, Case B).
//
// Differences from the row-per-warp kernel, both measured on GB300:
//
//  * Dense access order.  The rows of a row class are dealt to its CTAs
//    round-robin and each CTA streams its rows in tiles of RT, so local tile
//    g of every CTA covers one contiguous block of rows: at any moment the
//    whole GPU streams one narrow window of B (the order a grid-stride copy
//    uses), instead of thousands of unrelated row streams spread over the
//    matrix, and CTA loads differ by at most one row.
//  * One code path for any alignment.  The rows of B start at element
//    offset (base + i*ldb) mod 8 inside a 16-byte block (ldb = the row
//    stride, k unless the caller passes a padded one), which depends only on
//    i mod 8.  CTAs are assigned one residue class of rows each, so every
//    row a CTA reads has the same offset `off`: the CTA stages its k-segment
//    of a shifted by `off` once, and row blocks then line up with staged
//    16-byte vectors of a.  The only extra work for k % 8 != 0 is masking
//    the first and last block of each row (elements of neighbouring rows).
//  * Rows are split into S slices of L blocks (one warp per slice, each lane
//    streaming up to U 16-byte blocks, R rows side by side for short rows);
//    the S slice sums of a row are combined in shared memory in slice order
//    after a named barrier among the S warps of that row team (double-
//    buffered, so one barrier per tile suffices).
#pragma once

#include "gemv_kernels.cuh"

namespace gemvk {

__device__ __forceinline__ void team_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Ask the L2 to fetch [p, p + bytes) (16-byte aligned, multiple of 16) from
// HBM; no registers are held and nothing is returned.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Source vector q of the segment: a[j0 + 8q .. j0 + 8q + 7], zero outside
// the segment's columns [0, len).  `aj` = a + j0; `vec_ok`: aj is 16-byte
// aligned, so whole vectors can be loaded at once.
__device__ __forceinline__ uint4 a_vec(const uint16_t *aj, int64_t q, int64_t len, bool vec_ok) {
  const int64_t jb = 8 * q;
  if (q < 0 || jb >= len) return zero4();
  if (vec_ok && jb + 8 <= len) return __ldg(reinterpret_cast<const uint4 *>(aj + jb));
  uint32_t w[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int64_t j_lo = jb + 2 * h, j_hi = jb + 2 * h + 1;
    const uint32_t lo = (j_lo < len) ? (uint32_t)__ldg(aj + j_lo) : 0u;
    const uint32_t hi = (j_hi < len) ? (uint32_t)__ldg(aj + j_hi) : 0u;
    w[h] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// as4[q] = elements [SH, SH + 8) of source vectors (q - 1) ++ q, i.e. the
// segment shifted right by off = 8 - SH elements.  Unshifted (SH == 8), a
// thread's loads of a go out two at a time before either is stored, so the
// staging pays one L2 round trip per pair of vectors (measured ~1 % faster
// per call back to back at k >= 7168; the shifted loops, which need two
// source vectors per output, stay one vector at a time: batching them
// measured slower).
template <int SH>
__device__ __forceinline__ void stage_shift_loop(uint4 *as4, int nvec, const uint16_t *aj, int64_t len, bool vec_ok) {
  const int step = blockDim.x;
  int q = threadIdx.x;
  if constexpr (SH == 8) {
    for (; q + step < nvec; q += 2 * step) {
      const uint4 v0 = a_vec(aj, q, len, vec_ok);
      const uint4 v1 = a_vec(aj, q + step, len, vec_ok);
      as4[q] = v0;
      as4[q + step] = v1;
    }
  }
  for (; q < nvec; q += step) {
    const uint4 hi = a_vec(aj, q, len, vec_ok);
    if constexpr (SH == 8) {
      as4[q] = hi;
    } else {
      as4[q] = window<SH>(a_vec(aj, q - 1, len, vec_ok), hi);
    }
  }
}

// Stage columns [j0, j0 + len) of a, shifted right by `off` elements:
// as[x] = a[j0 + x - off] for off <= x < off + len, 0 for other x < as_elems.
// Block t of a row that starts at offset `off` then multiplies as4[t].
// Built from whole 16-byte loads of a plus a register shift (one code path
// per offset, chosen once per CTA).
__device__ __forceinline__ void stage_a_shifted(const Params &p, uint4 *as4, int64_t j0, int64_t len, int off) {
  const int nvec = p.as_elems >> 3;
  const uint16_t *aj = p.a + j0;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(aj) & 15u) == 0;
  switch (8 - off) {
    case 1: stage_shift_loop<1>(as4, nvec, aj, len, vec_ok); break;
    case 2: stage_shift_loop<2>(as4, nvec, aj, len, vec_ok); break;
    case 3: stage_shift_loop<3>(as4, nvec, aj, len, vec_ok); break;
    case 4: stage_shift_loop<4>(as4, nvec, aj, len, vec_ok); break;
    case 5: stage_shift_loop<5>(as4, nvec, aj, len, vec_ok); break;
    case 6: stage_shift_loop<6>(as4, nvec, aj, len, vec_ok); break;
    case 7: stage_shift_loop<7>(as4, nvec, aj, len, vec_ok); break;
    default: stage_shift_loop<8>(as4, nvec, aj, len, vec_ok); break;
  }
}

// Issue this lane's loads of one step of a row slice: blocks t + 32u
// (u < U) of the R rows, predicated on t + 32u < t1 and the row being real.
template <int U, int R>
__device__ __forceinline__ void tile_issue(const uint4 *bal, const int64_t (&g0)[R], const bool (&valid)[R],
                                           int t, int t1, uint4 (&bv)[U][R]) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int tt = t + 32 * u;
#pragma unroll
    for (int r = 0; r < R; ++r) bv[u][r] = (tt < t1 && valid[r]) ? ldg_stream(bal + g0[r] + tt) : zero4();
  }
}

// Multiply-accumulate one step's blocks with the staged (pre-shifted) a.
// No masking: for an unaligned row the first and last block also hold
// elements of the neighbouring rows, but the staged a is zero at those
// positions, so they add exactly 0 -- unless they are Inf or NaN (0 * Inf =
// NaN).  That case can only turn the sum NaN and is redone by tile_redo().
template <class T, int U, int R, int NA>
__device__ __forceinline__ void tile_consume(const uint4 *as4, const uint4 (&bv)[U][R], int t, int t1,
                                             float (&acc)[R][NA][2]) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int tt = t + 32 * u;
    if (tt < t1) {
      float af[8];
      widen8<T>(as4[tt], af);
#pragma unroll
      for (int r = 0; r < R; ++r) fma8<T, NA>(bv[u][r], af, acc[r]);
    }
  }
}

// The slow path of an unaligned row slice whose fast sum came out NaN:
// stream the slice [t0, t1) of one row again with the neighbouring rows'
// elements of the edge blocks (0 and nt - 1) zeroed.  Warp-uniform.
template <class T>
__device__ __forceinline__ float tile_redo(const uint4 *bal, const uint4 *as4, int64_t g0, int t0, int t1, int nt,
                                        int off, int last_hi, int lane) {
  float acc[1][2] = {{0.f, 0.f}};
  for (int t = t0 + lane; t < t1; t += 32) {
    uint4 b = ldg_stream(bal + g0 + t);
    if (t == 0 || t == nt - 1) b = keep_range(b, t == 0 ? off : 0, t == nt - 1 ? last_hi : 8);
    float af[8];
    widen8<T>(as4[t], af);
    fma8<T, 1>(b, af, acc);
  }
  return warp_sum(acc_total<1>(acc));
}

// Grid: blockIdx.x = c * sg + gs, c in [0, C) with C = p.nrb.  ALIGNED
// (k % 8 == 0 and B 16-byte aligned) uses one row class; otherwise 8 classes
// (C must be a multiple of 8), CTA c serving class c % 8.
template <class T, bool OUT_F32, int U, int R, bool ALIGNED, bool EPI>
__global__ void __launch_bounds__(kMaxThreads, 2) gemv_tiles_kernel(Params p) {
  extern __shared__ __align__(16) uint4 smem4[];
  uint4 *as4 = smem4;
  float *ps = reinterpret_cast<float *>(smem4 + (p.as_elems >> 3));  // [2][W * R]
  constexpr int NA = (R == 1) ? 2 : 1;  // accumulator pairs per row

  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gs = blockIdx.x % p.sg;
  const int c = blockIdx.x / p.sg;
  constexpr int NCLS = ALIGNED ? 1 : 8;
  const int cls = c % NCLS, cq = c / NCLS, Cq = p.nrb / NCLS;
  const int64_t j0 = (int64_t)gs * p.kseg;
  const int64_t len = (p.k - j0 < p.kseg) ? (p.k - j0) : p.kseg;
  // rows of this class: i = NCLS * j + cls, 0 <= j < nr
  const int64_t nr = (p.n > cls) ? (p.n - cls + NCLS - 1) / NCLS : 0;
  const int off = ALIGNED ? 0 : (int)(((int64_t)p.base_off + j0 + (int64_t)cls * (p.ldb & 7)) & 7);
  const int nt = (int)((off + len + 7) >> 3);
  const int last_hi = (int)(len + off - 8 * (int64_t)(nt - 1));

  const uint4 *bal = reinterpret_cast<const uint4 *>(reinterpret_cast<uintptr_t>(p.B) & ~(uintptr_t)15);
  const int S = p.sw, slots = W / S, slot = warp / S, s = warp % S;
  const int RT = slots * R;  // rows per tile
  const int L = (nt + S - 1) / S;
  const int t0 = s * L < nt ? s * L : nt;
  const int t1 = t0 + L < nt ? t0 + L : nt;
  // Rows of the class are dealt to the class's Cq CTAs round-robin: this CTA
  // owns class rows j = cq + Cq*m, m < nloc (so CTA loads differ by at most
  // one row), streamed as local tiles of RT consecutive m.  Local tile g of
  // every CTA covers class rows [Cq*RT*g, Cq*RT*(g+1)): one contiguous window
  // of B at a time across the GPU.
  const int64_t nloc = nr > cq ? (nr - cq + Cq - 1) / Cq : 0;
  const int64_t ngroups = (nloc + RT - 1) / RT;
  if (ngroups == 0) {  // no rows for this CTA (a short row class): no staging, no loads
    allow_dependents();
    return;
  }
  auto row_of = [&](int64_t m) -> int64_t { return NCLS * (cq + (int64_t)Cq * m) + cls; };

  auto rows_of = [&](int64_t g, int64_t (&g0)[R], bool (&valid)[R]) {
    const int64_t mb = g * RT + (int64_t)slot * R;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      valid[r] = (mb + r) < nloc;
      g0[r] = valid[r] ? (((int64_t)p.base_off + row_of(mb + r) * p.ldb + j0) >> 3) : 0;
    }
  };

  // Bulk L2 prefetch of this warp's row slices of tile g (lane r < R
  // issues row r's), `pf` rounds ahead of the tile being streamed.
  const int pf = (p.flags >> kFlagL2Shift) & 3;
  auto prefetch_tile = [&](int64_t g) {
    if (g < ngroups && lane < R && t1 > t0) {
      const int64_t m = g * RT + (int64_t)slot * R + lane;
      if (m < nloc) {
        const int64_t gb = ((int64_t)p.base_off + row_of(m) * p.ldb + j0) >> 3;
        prefetch_l2(bal + gb + t0, (uint32_t)(t1 - t0) * 16u);
      }
    }
  };

  // Under a programmatic dependent launch with kFlagPrefetchB the first
  // tile's first loads go out before the preceding kernel has finished (B
  // is then promised read-only), and a is staged after them.  Without that
  // promise (kFlagL2First), each warp only asks L2 for the blocks of its
  // first loads before waiting (a prefetch reads nothing into the kernel,
  // and L2 is where the preceding kernel's writes land, so no write can be
  // missed); after the wait a is staged first and the first loads, L2 hits
  // by then, go out behind it.  a is read by every CTA at once; issued
  // behind eight B loads per lane its loads queued for ~3 us after the
  // wait, and staging it first measured 3-16 % faster per call back to back
  // (7168 x 16384 33.0 -> 31.8 us, 4096 x 4096 7.10 -> 6.33), faster as
  // plain and isolated launches too.  a and c are touched only after
  // wait_for_predecessor().
  allow_dependents();
  const bool early = (p.flags & kFlagPrefetchB) != 0;
  if (!early) {
    if ((p.flags & kFlagL2First) && lane < R && t1 > t0 && (int64_t)slot * R + lane < nloc) {
      const int64_t gb = ((int64_t)p.base_off + row_of((int64_t)slot * R + lane) * p.ldb + j0) >> 3;
      const int nb = (t1 - t0) < 32 * U ? (t1 - t0) : 32 * U;
      prefetch_l2(bal + gb + t0, (uint32_t)nb * 16u);
    }
    wait_for_predecessor();
    stage_a_shifted(p, as4, j0, len, off);
  }
  uint4 bv[U][R];
  bool prefetched = false;
  if (ngroups > 0) {
    int64_t g0[R];
    bool valid[R];
    rows_of(0, g0, valid);
    tile_issue<U, R>(bal, g0, valid, t0 + lane, t1, bv);
    prefetched = true;
    // Also ask L2 for the blocks of the warp's second step (the next 32*U
    // blocks of its rows' slices), so that HBM keeps streaming while the
    // first step is consumed.  With B promised unwritten this goes out
    // before the wait on the predecessor; otherwise (after the wait, behind
    // the staging of a and the first step's loads: issued ahead of the
    // staging it delayed a and measured 2-4 % slower) only when the CTA
    // streams more than one row tile (4096 x 4096, a single tile per CTA,
    // measured 6 % slower with it).
    // Lane r issues row r's.  A slice of one step prefetches nothing
    // (asking for the first step of the next tile's rows instead measured
    // 2-4 % slower at k = 1000).
    if (early || ngroups > 1) {
      const int b0 = t0 + 32 * U;
      const int b1 = (b0 + 32 * U) < t1 ? (b0 + 32 * U) : t1;
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (lane == r && valid[r] && b1 > b0) prefetch_l2(bal + g0[r] + b0, (uint32_t)(b1 - b0) * 16u);
    }
  }
  for (int m = 1; m <= pf; ++m) prefetch_tile(m);
  // With B promised, a is staged here: before the wait only when the
  // caller promised that the predecessor does not write it either
  // (kFlagPrefetchA), else after it.  c is always written
  // after the wait.  With kFlagDeferStores (only set with kFlagPrefetchA)
  // the CTA's row results are kept in shared memory and written after a
  // single wait at the end: the whole stream of B then overlaps the
  // preceding kernel's drain.
  const bool early_a = early && (p.flags & kFlagPrefetchA) != 0;
  const bool defer = early_a && (p.flags & kFlagDeferStores) != 0;
  float *res = ps + 2 * W * R;  // [nloc] row results when deferring
  if (early && !early_a) wait_for_predecessor();
  if (early) stage_a_shifted(p, as4, j0, len, off);
  __syncthreads();
  if (early_a && !defer) wait_for_predecessor();

  int buf = 0;
  for (int64_t g = 0; g < ngroups; ++g) {
    int64_t g0[R];
    bool valid[R];
    rows_of(g, g0, valid);
    if (pf > 0 && g > 0) prefetch_tile(g + pf);
    float acc[R][NA][2];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int q = 0; q < NA; ++q) acc[r][q][0] = acc[r][q][1] = 0.f;
    }
    for (int t = t0 + lane; t < t1; t += 32 * U) {
      if (!prefetched) tile_issue<U, R>(bal, g0, valid, t, t1, bv);
      prefetched = false;
      // A last step of at most one block per lane (the extra edge block of
      // an unaligned row makes a slice 32*U*m + 1 blocks long) is folded
      // into this one: its loads go out with this step's, saving a whole
      // memory round trip.  The blocks are added in the same order as in a
      // step of their own.
      const int tx = t + 32 * U;
      const int rem = t1 - (tx - lane);  // blocks after this step (warp-uniform)
      if (R <= 2 && rem > 0 && rem <= 32) {
        uint4 bx[R];
#pragma unroll
        for (int r = 0; r < R; ++r) bx[r] = (tx < t1 && valid[r]) ? ldg_stream(bal + g0[r] + tx) : zero4();
        tile_consume<T, U, R, NA>(as4, bv, t, t1, acc);
        if (tx < t1) {
          float af[8];
          widen8<T>(as4[tx], af);
#pragma unroll
          for (int r = 0; r < R; ++r) fma8<T, NA>(bx[r], af, acc[r]);
        }
        break;
      }
      tile_consume<T, U, R, NA>(as4, bv, t, t1, acc);
    }
    prefetched = false;
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = warp_sum(acc_total<NA>(acc[r]));
    if constexpr (!ALIGNED) {
      if (t0 == 0 || t1 == nt) {  // this slice holds a row edge
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (valid[r] && isnan(v[r])) v[r] = tile_redo<T>(bal, as4, g0[r], t0, t1, nt, off, last_hi, lane);
      }
    }
    const int64_t mb = g * RT + (int64_t)slot * R;
    if (S == 1) {
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (valid[r]) {
            if (defer) {
              res[mb + r] = v[r];
            } else {
              store_out<T, OUT_F32, EPI>(p, gs, row_of(mb + r), v[r]);
            }
          }
      }
    } else {
      float *pb = ps + buf * (W * R);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) pb[(slot * R + r) * S + s] = v[r];
      }
      team_barrier(1 + slot, S * 32);
      if (s == 0 && lane < R) {
        const int64_t m = mb + lane;
        if (m < nloc) {
          float sum = 0.f;
          for (int s2 = 0; s2 < S; ++s2) sum += pb[(slot * R + lane) * S + s2];
          if (defer) {
            res[m] = sum;
          } else {
            store_out<T, OUT_F32, EPI>(p, gs, row_of(m), sum);
          }
        }
      }
      buf ^= 1;
    }
  }
  if (defer) {
    wait_for_predecessor();
    __syncthreads();
    for (int64_t m = threadIdx.x; m < nloc; m += blockDim.x) store_out<T, OUT_F32, EPI>(p, gs, row_of(m), res[m]);
  }
}

}  // namespace gemvk

// Instantiations of the tiles kernel for one input type: (U, R) in
// {(8,1), (4,1), (4,2), (2,4)}, aligned or not, output same type or fp32,
// with or without the fused epilogue.
#define GEMV_TILES_CASES(T, OF, AL, EP)                                     \
  if (U == 8 && R == 1) return gemv_tiles_kernel<T, OF, 8, 1, AL, EP>;      \
  if (U == 4 && R == 1) return gemv_tiles_kernel<T, OF, 4, 1, AL, EP>;      \
  if (U == 4 && R == 2) return gemv_tiles_kernel<T, OF, 4, 2, AL, EP>;      \
  if (U == 2 && R == 4) return gemv_tiles_kernel<T, OF, 2, 4, AL, EP>;

#define GEMV_TILES_BY_ALIGN(T, OF, EP)                                       \
  if (aligned) { GEMV_TILES_CASES(T, OF, true, EP) } else { GEMV_TILES_CASES(T, OF, false, EP) }

#define GEMV_DEFINE_TILES_TABLE(T, SUFFIX)                                             \
  namespace gemvk {                                                                    \
  MainKernel tiles_kernel_##SUFFIX(int out_f32, int aligned, int R, int U, int epi) {  \
    if (out_f32) {                                                                     \
      if (epi) { GEMV_TILES_BY_ALIGN(T, true, true) } else { GEMV_TILES_BY_ALIGN(T, true, false) } \
    } else {                                                                           \
      if (epi) { GEMV_TILES_BY_ALIGN(T, false, true) } else { GEMV_TILES_BY_ALIGN(T, false, false) } \
    }                                                                                  \
    return nullptr;                                                                    \
  }                                                                                    \
  }

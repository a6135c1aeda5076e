// "Bulk" GEMV kernel for sm_103a: the tiles kernel's work split with B
// staged through shared memory by the Tensor Memory Accelerator instead of
// being loaded into registers.
//
// The pages pipeline B through shared memory with cp.async and 1-3 stages
// (TileLang Case Studies, Case B.1 "O3 Pipelined B Loads"): it helped at
// k = 7168 and hurt at k = 16384 on H200.  The sm_103a form of that idea is a
// 1-D bulk asynchronous copy (cp.async.bulk global -> shared, completion
// counted in bytes on an mbarrier), which needs one issuing thread and no
// registers per byte in flight:
//
//  * Each warp owns a ring of NS buffers of 32*U 16-byte blocks.  Its
//    sequence of work is the chunks of its row slices -- row slice after row
//    slice, each cut into pieces of at most 32*U blocks -- and chunk c goes
//    to buffer c mod NS.  Lane 0 issues the first NS chunks up front; after
//    the warp has consumed chunk c, lane 0 refills that buffer with chunk
//    c + NS.  So NS chunks are in flight while a warp computes, without any
//    cross-warp handshake.
//  * Consuming a chunk: every lane waits on the buffer's mbarrier phase, then
//    multiplies blocks lane + 32u of the buffer with the staged (pre-shifted)
//    a, exactly as the tiles kernel does with its registers.
//  * Rows, classes, slices, the shifted a, the NaN-triggered edge redo and the
//    slice combination are the tiles kernel's (R = 1).
//  * Every wait polls a bounded number of times.  A warp whose wait gives up
//    stops issuing, keeps going through its row tiles (so the named barriers
//    its team shares still complete), writes NaN for its rows, waits
//    (bounded) for the copies it has in flight and counts one timeout in a
//    device word the host can read.  No multicast.
#pragma once

#include "gemv_tiles.cuh"

namespace gemvk {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One arrival expected per phase: lane 0's arrive.expect_tx.
__device__ __forceinline__ void ring_bar_init(uint64_t *bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void ring_bar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Refill one ring buffer: announce `bytes` on its mbarrier, then start the
// bulk copy of `bytes` (a multiple of 16) from global `src` (16-byte aligned)
// into shared `dst` (16-byte aligned); the copy's completion finishes the
// phase.  The proxy fence orders the warp's earlier generic reads of the
// buffer (made visible to this lane by __syncwarp) before the async write.
__device__ __forceinline__ void ring_fill(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool ring_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      "  .reg .pred P;\n"
      "  mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, P;\n"
      "}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with parity `parity` to complete, polling at most
// `polls` times.  Returns false if it did not complete.
__device__ __forceinline__ bool ring_wait(uint64_t *bar, uint32_t parity, int polls) {
  for (int i = 0; i < polls; ++i)
    if (ring_try_wait(bar, parity)) return true;
  return false;
}

// Grid and row mapping: as gemv_tiles_kernel with R = 1.
template <class T, bool OUT_F32, int U, bool ALIGNED, bool EPI>
__global__ void __launch_bounds__(kMaxThreads, 2) gemv_bulk_kernel(const Params p) {
  extern __shared__ __align__(16) uint4 smem4[];
  constexpr int SB = 32 * U;  // 16-byte blocks per ring buffer
  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = p.stages;
  uint4 *as4 = smem4;
  float *ps = reinterpret_cast<float *>(smem4 + (p.as_elems >> 3));  // [2][W]
  char *ring_base = reinterpret_cast<char *>(smem4) + bulk_ring_offset(p.as_elems, W);
  uint4 *ring = reinterpret_cast<uint4 *>(ring_base) + (size_t)warp * NS * SB;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring_base + (size_t)W * NS * SB * 16) + warp * NS;

  const int gs = blockIdx.x % p.sg;
  const int c = blockIdx.x / p.sg;
  constexpr int NCLS = ALIGNED ? 1 : 8;
  const int cls = c % NCLS, cq = c / NCLS, Cq = p.nrb / NCLS;
  const int64_t j0 = (int64_t)gs * p.kseg;
  const int64_t len = (p.k - j0 < p.kseg) ? (p.k - j0) : p.kseg;
  const int64_t nr = (p.n > cls) ? (p.n - cls + NCLS - 1) / NCLS : 0;
  const int off = ALIGNED ? 0 : (int)(((int64_t)p.base_off + j0 + (int64_t)cls * (p.ldb & 7)) & 7);
  const int nt = (int)((off + len + 7) >> 3);
  const int last_hi = (int)(len + off - 8 * (int64_t)(nt - 1));

  const uint4 *bal = reinterpret_cast<const uint4 *>(reinterpret_cast<uintptr_t>(p.B) & ~(uintptr_t)15);
  const int S = p.sw, slots = W / S, slot = warp / S, s = warp % S;
  const int RT = slots;  // rows per tile
  const int L = (nt + S - 1) / S;
  const int t0 = s * L < nt ? s * L : nt;
  const int t1 = t0 + L < nt ? t0 + L : nt;
  const int64_t nloc = nr > cq ? (nr - cq + Cq - 1) / Cq : 0;
  const int64_t ngroups = (nloc + RT - 1) / RT;
  if (ngroups == 0) {  // no rows for this CTA (a short row class): no staging, no loads
    allow_dependents();
    return;
  }
  auto row_of = [&](int64_t m) -> int64_t { return NCLS * (cq + (int64_t)Cq * m) + cls; };
  auto block_of = [&](int64_t g) -> int64_t {  // first 16-byte block of row slice g's row
    return ((int64_t)p.base_off + row_of(g * RT + slot) * p.ldb + j0) >> 3;
  };

  // This warp's chunks: tiles g < gv hold a row for it; each row slice is
  // nst chunks.
  const int nst = (t1 - t0 + SB - 1) / SB;
  const int64_t gv = nloc > slot ? (nloc - slot + RT - 1) / RT : 0;
  const int64_t total = gv * nst;

  if (lane == 0) {
    for (int i = 0; i < NS; ++i) ring_bar_init(&bars[i]);
    ring_bar_init_fence();
  }
  __syncwarp();

  // Issue cursor (lane 0 only): next chunk ic = ig * nst + ist, into buffer ib.
  int64_t ic = 0, ig = 0;
  int ist = 0, ib = 0;
  auto issue_next = [&]() {
    const int tb = t0 + ist * SB;
    const int nb = (t1 - tb) < SB ? (t1 - tb) : SB;
    ring_fill(ring + (size_t)ib * SB, bal + block_of(ig) + tb, (uint32_t)nb * 16u, &bars[ib]);
    ++ic;
    if (++ib == NS) ib = 0;
    if (++ist == nst) {
      ist = 0;
      ++ig;
    }
  };

  // Under a programmatic dependent launch with kFlagPrefetchB the first NS
  // chunks go out before the preceding kernel has finished (B is then
  // promised read-only), and a is staged after them.  Without that promise
  // (kFlagL2First), lane 0 only asks L2 for those chunks' blocks before
  // waiting (a prefetch reads nothing into the kernel); after the wait a is
  // staged first and the chunks go out behind it, as in the tiles kernel
  // (measured 0.5-1.1 % faster per call here).
  allow_dependents();
  const bool early = (p.flags & kFlagPrefetchB) != 0;
  if (!early) {
    if ((p.flags & kFlagL2First) && lane == 0 && gv > 0 && t1 > t0) {
      const int nb = (t1 - t0) < NS * SB ? (t1 - t0) : NS * SB;
      prefetch_l2(bal + block_of(0) + t0, (uint32_t)nb * 16u);
    }
    wait_for_predecessor();
    stage_a_shifted(p, as4, j0, len, off);
  }
  if (lane == 0) {
    while (ic < total && ic < NS) issue_next();
  }
  const bool early_a = early && (p.flags & kFlagPrefetchA) != 0;
  if (early && !early_a) wait_for_predecessor();
  if (early) stage_a_shifted(p, as4, j0, len, off);
  __syncthreads();
  if (early_a) wait_for_predecessor();

  int cb = 0;          // buffer of the next chunk to consume
  uint32_t cpar = 0;   // parity of that buffer's phase
  bool bad = false;    // a wait gave up (warp-uniform)
  int64_t cfail = 0;   // first chunk not consumed after giving up
  int fb = 0;          // its buffer
  int buf = 0;
  for (int64_t g = 0; g < ngroups; ++g) {
    const bool valid = g < gv;
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (valid) {
      for (int st = 0; st < nst; ++st) {
        if (!bad) {
          const bool ok = __all_sync(0xffffffffu, ring_wait(&bars[cb], cpar, p.wait_polls));
          if (!ok) {
            bad = true;
            cfail = g * nst + st;
            fb = cb;
          }
        }
        if (!bad) {
          const uint4 *stg = ring + (size_t)cb * SB;
          const int tb = t0 + st * SB;
          const int nb = (t1 - tb) < SB ? (t1 - tb) : SB;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int x = lane + 32 * u;
            if (x < nb) {
              float af[8];
              widen8<T>(as4[tb + x], af);
              fma8<T, 2>(stg[x], af, acc);
            }
          }
          __syncwarp();
          if (lane == 0 && ic < total) issue_next();  // chunk + NS, into buffer cb
        }
        if (++cb == NS) {
          cb = 0;
          cpar ^= 1u;
        }
      }
    }
    float v = warp_sum(acc_total<2>(acc));
    if (bad) {
      v = __int_as_float(0x7fc00000);
    } else if constexpr (!ALIGNED) {
      if (valid && (t0 == 0 || t1 == nt) && isnan(v)) v = tile_redo<T>(bal, as4, block_of(g), t0, t1, nt, off, last_hi, lane);
    }
    if (S == 1) {
      if (lane == 0 && valid) store_out<T, OUT_F32, EPI>(p, gs, row_of(g * RT + slot), v);
    } else {
      float *pb = ps + buf * W;
      if (lane == 0) pb[slot * S + s] = v;
      team_barrier(1 + slot, S * 32);
      if (s == 0 && lane == 0 && valid) {
        float sum = 0.f;
        for (int s2 = 0; s2 < S; ++s2) sum += pb[slot * S + s2];
        store_out<T, OUT_F32, EPI>(p, gs, row_of(g * RT + slot), sum);
      }
      buf ^= 1;
    }
  }
  if (bad && lane == 0) {
    // Copies issued but not consumed, [cfail, ic), one per buffer at most:
    // wait for each (bounded) before the CTA's shared memory goes away.  If
    // one of these waits runs out too, a copy may still be in flight when
    // the CTA exits: that is recorded apart, in the counter's top bit.
    int b = fb;
    bool drained = true;
    for (int64_t j = cfail; j < ic; ++j) {
      if (!ring_wait(&bars[b], (uint32_t)((j / NS) & 1), kWaitPolls)) drained = false;
      if (++b == NS) b = 0;
    }
    atomicAdd(p.timeouts, 1u);
    if (!drained) atomicOr(p.timeouts, kDrainTimeoutBit);
  }
}

}  // namespace gemvk

// Instantiations of the bulk kernel for one input type: U in {4, 8}, aligned
// or not, output same type or fp32, with or without the fused epilogue.
#define GEMV_BULK_BY_U(T, OF, AL, EP)                              \
  if (U == 8) return gemv_bulk_kernel<T, OF, 8, AL, EP>;           \
  if (U == 4) return gemv_bulk_kernel<T, OF, 4, AL, EP>;

#define GEMV_BULK_BY_ALIGN(T, OF, EP) \
  if (aligned) { GEMV_BULK_BY_U(T, OF, true, EP) } else { GEMV_BULK_BY_U(T, OF, false, EP) }

#define GEMV_DEFINE_BULK_TABLE(T, SUFFIX)                                                      \
  namespace gemvk {                                                                            \
  MainKernel bulk_kernel_##SUFFIX(int out_f32, int aligned, int U, int epi) {                  \
    if (out_f32) {                                                                             \
      if (epi) { GEMV_BULK_BY_ALIGN(T, true, true) } else { GEMV_BULK_BY_ALIGN(T, true, false) } \
    } else {                                                                                   \
      if (epi) { GEMV_BULK_BY_ALIGN(T, false, true) } else { GEMV_BULK_BY_ALIGN(T, false, false) } \
    }                                                                                          \
    return nullptr;                                                                            \
  }                                                                                            \
  }

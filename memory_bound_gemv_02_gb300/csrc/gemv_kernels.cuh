// Streaming GEMV kernels for sm_103a: c = B @ a, B (n, k) row-major,
// fp16/bf16 inputs, fp32 accumulation (TileLang Case Studies, Case B).
//
// Design (a GB300-first restatement of the pages' coalesced "O1" layout,
// Case B "Fix (O1)", where the fast thread index walks k within one row):
//
//  * A warp owns rows.  Its 32 lanes read consecutive 16-byte vectors of the
//    same row, so one warp-wide load covers 512 contiguous bytes: every
//    32-byte sector fetched is fully used (the 32-way strided pattern of
//    Case B "Root Cause" cannot occur).  Loads bypass L1 (B is read once).
//  * Each lane issues U loads back to back (R rows x U vectors in flight),
//    so a resident warp keeps 8 x 16 B per lane outstanding.
//  * The CTA's k-segment of a is staged once in shared memory (Case B.2's
//    "O2", here needed because the general variant realigns it per row);
//    each 16-byte vector of a read from shared memory is reused for R rows.
//  * Partial sums stay in fp32 registers (4 independent accumulators per
//    row), are reduced across the warp with xor shuffles, across warps of a
//    CTA in shared memory (warp split), and across CTAs through a workspace
//    plus a second kernel (grid split / split-K, as in Case C's split-K +
//    reduce pair).  Every combination step runs in a fixed order.
//  * Rows whose start is not 16-byte aligned (k % 8 != 0, or an offset B)
//    read the aligned 16-byte blocks that cover the row, zero the elements
//    that belong to neighbouring rows, and shift the staged a by the row's
//    offset in registers (a byte permute selected by a template constant).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gemv_internal.h"

namespace gemvk {

// ----------------------------------------------------------------- types --

struct F16 {
  static __device__ __forceinline__ float2 pair(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
  }
  static __device__ __forceinline__ uint16_t from_float(float x) {
    return __half_as_ushort(__float2half_rn(x));
  }
  static __device__ __forceinline__ float to_float(uint16_t h) { return __half2float(__ushort_as_half(h)); }
};

struct BF16 {
  // bf16 is the upper half of an fp32: widening is a shift / mask.
  static __device__ __forceinline__ float2 pair(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ uint16_t from_float(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
  static __device__ __forceinline__ float to_float(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
};

// --------------------------------------------------------------- memory --

// 16-byte streaming load of data read exactly once: non-coherent path,
// no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 zero4() { return make_uint4(0u, 0u, 0u, 0u); }

// Programmatic dependent launch.  allow_dependents(): the next kernel on the
// stream (if launched with the programmatic-serialization attribute) may be
// scheduled once every CTA of this grid has executed it or exited.
// wait_for_predecessor(): blocks until the preceding grid has completed and
// its memory is visible; a no-op when this grid was launched normally.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_for_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------ arithmetic --

// Widen a 16-byte vector of a (8 elements) to fp32.
template <class T>
__device__ __forceinline__ void widen8(const uint4 &v, float (&f)[8]) {
  float2 p0 = T::pair(v.x), p1 = T::pair(v.y), p2 = T::pair(v.z), p3 = T::pair(v.w);
  f[0] = p0.x; f[1] = p0.y; f[2] = p1.x; f[3] = p1.y;
  f[4] = p2.x; f[5] = p2.y; f[6] = p3.x; f[7] = p3.y;
}

// Packed fp32x2 FMA measured no faster than two fmaf on GB300 for this
// kernel (the pair packing costs what the pairing saves); off by default.
#ifndef GEMV_USE_FFMA2
#define GEMV_USE_FFMA2 0
#endif

// Two independent fp32 fused multiply-adds in one instruction (sm_100+):
// acc.x = fma(b.x, a.x, acc.x), acc.y = fma(b.y, a.y, acc.y), each rounded
// once exactly as fmaf.
__device__ __forceinline__ void ffma2(float &acc_x, float &acc_y, float b_x, float b_y, float a_x, float a_y) {
#if GEMV_USE_FFMA2
  unsigned long long acc, b, a;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(acc_x), "f"(acc_y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b_x), "f"(b_y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a_x), "f"(a_y));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(b), "l"(a));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(acc_x), "=f"(acc_y) : "l"(acc));
#else
  acc_x = fmaf(b_x, a_x, acc_x);
  acc_y = fmaf(b_y, a_y, acc_y);
#endif
}

// Multiply-accumulate one 16-byte vector of B (8 elements) with the
// matching widened a elements.  NA accumulator pairs (x for even, y for odd
// elements): element pair q goes to pair (q % NA); 4 pairs give eight
// independent chains of one.
template <class T, int NA>
__device__ __forceinline__ void fma8(const uint4 &b, const float (&af)[8], float (&acc)[NA][2]) {
  const float2 p0 = T::pair(b.x), p1 = T::pair(b.y), p2 = T::pair(b.z), p3 = T::pair(b.w);
  ffma2(acc[0 % NA][0], acc[0 % NA][1], p0.x, p0.y, af[0], af[1]);
  ffma2(acc[1 % NA][0], acc[1 % NA][1], p1.x, p1.y, af[2], af[3]);
  ffma2(acc[2 % NA][0], acc[2 % NA][1], p2.x, p2.y, af[4], af[5]);
  ffma2(acc[3 % NA][0], acc[3 % NA][1], p3.x, p3.y, af[6], af[7]);
}

// Sum of the NA accumulator pairs (fixed order).
template <int NA>
__device__ __forceinline__ float acc_total(const float (&acc)[NA][2]) {
  float v = acc[0][0] + acc[0][1];
#pragma unroll
  for (int q = 1; q < NA; ++q) v += acc[q][0] + acc[q][1];
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Elements [SH, SH + 8) of the 16 elements lo ++ hi (SH in 1..8), as one
// 16-byte vector.  SH is a compile-time constant, so this is register
// selection plus (for odd SH) one byte permute per word.
template <int SH>
__device__ __forceinline__ uint4 window(const uint4 &lo, const uint4 &hi) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if constexpr ((SH & 1) == 0) {
      o[q] = w[SH / 2 + q];
    } else {
      // upper half of word (SH-1)/2+q, lower half of the next word
      o[q] = __byte_perm(w[(SH - 1) / 2 + q], w[(SH + 1) / 2 + q], 0x5432);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Keep elements p with lo <= p < hi of an 8-element vector, zero the rest.
__device__ __forceinline__ uint4 keep_range(uint4 v, int lo, int hi) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e0 = 2 * q, e1 = 2 * q + 1;
    uint32_t m = ((e0 >= lo && e0 < hi) ? 0x0000ffffu : 0u) | ((e1 >= lo && e1 < hi) ? 0xffff0000u : 0u);
    w[q] &= m;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ------------------------------------------------------------- staging --

// as[x] = a[j0 + x - 8] for 8 <= x < 8 + len, 0 for every other x < as_elems.
// The 8 leading zeros let the general variant read one vector before the
// segment's first column.
__device__ __forceinline__ void stage_a(const Params &p, uint4 *as4, int64_t j0, int64_t len) {
  const int nvec = p.as_elems >> 3;
  const uint16_t *aj = p.a + j0;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(aj) & 15u) == 0;
  for (int q = threadIdx.x; q < nvec; q += blockDim.x) {
    const int64_t jb = 8 * (int64_t)q - 8;  // segment column of element 0 of this vector
    uint4 v;
    if (vec_ok && jb >= 0 && jb + 8 <= len) {
      v = __ldg(reinterpret_cast<const uint4 *>(aj + jb));
    } else {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int64_t j_lo = jb + 2 * h, j_hi = jb + 2 * h + 1;
        const uint32_t lo = (j_lo >= 0 && j_lo < len) ? (uint32_t)__ldg(aj + j_lo) : 0u;
        const uint32_t hi = (j_hi >= 0 && j_hi < len) ? (uint32_t)__ldg(aj + j_hi) : 0u;
        w[h] = lo | (hi << 16);
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    as4[q] = v;
  }
}

// ---------------------------------------------------------------- output --

// The fused epilogue on a row total, in fp32: y = act(alpha * v + beta *
// bias[row]).  With alpha = 1, no bias and no activation it returns v
// unchanged.  The activations call CUDA's expf.
template <class T>
__device__ __forceinline__ float apply_epilogue(const Epilogue &ep, int64_t row, float v) {
  float y = ep.alpha * v;
  if (ep.bias != nullptr) {
    const float b = ep.bias_f32 ? static_cast<const float *>(ep.bias)[row]
                                : T::to_float(static_cast<const uint16_t *>(ep.bias)[row]);
    y = fmaf(ep.beta, b, y);
  }
  switch (ep.act) {
    case 1: y = y > 0.f ? y : 0.f; break;                // relu
    case 2: y = 1.f / (1.f + expf(-y)); break;           // sigmoid
    case 3: y = y / (1.f + expf(-y)); break;             // silu: y * sigmoid(y)
    default: break;
  }
  return y;
}

// Final store of a row (rounded once), or its fp32 partial under split-K
// (the epilogue then runs in the second pass).  EPI: the kernel was built
// with the fused epilogue; plain GEMVs launch the copy without it, so their
// streaming loop carries none of its code.
template <class T, bool OUT_F32, bool EPI = true>
__device__ __forceinline__ void store_out(const Params &p, int gs, int64_t row, float v) {
  if (p.sg > 1) {
    p.ws[(int64_t)gs * p.n + row] = v;
    return;
  }
  float y = v;
  if constexpr (EPI) {
    if (p.flags & kFlagEpilogue) y = apply_epilogue<T>(p.ep, row, v);
  }
  if (OUT_F32) {
    static_cast<float *>(p.c)[row] = y;
  } else {
    static_cast<uint16_t *>(p.c)[row] = T::from_float(y);
  }
}

// ------------------------------------------------------- row dot products --

// Aligned variant: R rows (i0 .. i0+R-1, those < r1) over segment vectors
// [t0, t1); each row starts on a 16-byte boundary.  Returns per-row sums
// (valid in every lane).
template <class T, int R, int U>
__device__ __forceinline__ void rows_aligned(const Params &p, const uint4 *as4, int64_t i0, int64_t r1,
                                             int64_t j0, int t0, int t1, int lane, float (&out)[R]) {
  // Called with i0 < r1.  Rows past r1 (only in the CTA's last group)
  // re-read row i0 and their sums are discarded.
  const uint4 *b0 = reinterpret_cast<const uint4 *>(p.B + i0 * p.ldb + j0);
  const int kv = (int)(p.ldb >> 3);  // row stride in 16-byte vectors
  int roff[R];
#pragma unroll
  for (int r = 0; r < R; ++r) roff[r] = (i0 + r < r1) ? r * kv : 0;
  // Independent fp32 accumulators: 4 for one row, 2 each for two rows, 1
  // each for four (the R rows already give independent chains).
  constexpr int NA = (R == 1) ? 2 : 1;  // accumulator pairs per row
  float acc[R][NA][2];
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int q = 0; q < NA; ++q) acc[r][q][0] = acc[r][q][1] = 0.f;
  }
  for (int t = t0 + lane; t < t1; t += 32 * U) {
    uint4 bv[U][R];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tt = t + 32 * u;
#pragma unroll
      for (int r = 0; r < R; ++r) bv[u][r] = (tt < t1) ? ldg_stream(b0 + roff[r] + tt) : zero4();
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tt = t + 32 * u;
      if (tt < t1) {
        float af[8];
        widen8<T>(as4[tt + 1], af);
#pragma unroll
        for (int r = 0; r < R; ++r) fma8<T, NA>(bv[u][r], af, acc[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) out[r] = warp_sum(acc_total<NA>(acc[r]));
}

// General variant, one row.  The row's segment spans global 16-byte blocks
// g0 .. g0 + nt - 1 of the aligned base `bal`; its first element sits at
// position `off` of block g0.  Element p of block t is column
// 8t + p - off of the segment, which is staged at as[8t + SH + p] with
// SH = 8 - off.  Blocks [t0, t1) are this warp's share.
template <class T, int SH, int U>
__device__ __forceinline__ void row_general(const uint4 *bal, const uint4 *as4, int64_t g0, int off, int64_t len,
                                            int nt, int t0, int t1, int lane, float (&acc)[2][2]) {
  const int last_hi = (int)(len + off - 8 * (int64_t)(nt - 1));  // valid elements of the last block
  for (int t = t0 + lane; t < t1; t += 32 * U) {
    uint4 bv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tt = t + 32 * u;
      bv[u] = (tt < t1) ? ldg_stream(bal + g0 + tt) : zero4();
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tt = t + 32 * u;
      if (tt < t1) {
        uint4 b = bv[u];
        if (tt == 0 || tt == nt - 1) b = keep_range(b, tt == 0 ? off : 0, tt == nt - 1 ? last_hi : 8);
        uint4 av;
        if constexpr (SH == 8) {
          av = as4[tt + 1];
        } else {
          av = window<SH>(as4[tt], as4[tt + 1]);
        }
        float af[8];
        widen8<T>(av, af);
        fma8<T, 2>(b, af, acc);
      }
    }
  }
}

template <class T, int U>
__device__ __forceinline__ float row_general_dispatch(const Params &p, const uint4 *as4, int64_t i, int64_t j0,
                                                      int64_t len, int s, int sw, int lane) {
  const uint4 *bal = reinterpret_cast<const uint4 *>(reinterpret_cast<uintptr_t>(p.B) & ~(uintptr_t)15);
  const int64_t e0 = (int64_t)p.base_off + i * p.ldb + j0;  // element index from the aligned base
  const int64_t g0 = e0 >> 3;
  const int off = (int)(e0 & 7);
  const int nt = (int)((off + len + 7) >> 3);
  const int t0 = (int)((int64_t)nt * s / sw), t1 = (int)((int64_t)nt * (s + 1) / sw);
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  switch (8 - off) {  // warp-uniform
    case 1: row_general<T, 1, U>(bal, as4, g0, off, len, nt, t0, t1, lane, acc); break;
    case 2: row_general<T, 2, U>(bal, as4, g0, off, len, nt, t0, t1, lane, acc); break;
    case 3: row_general<T, 3, U>(bal, as4, g0, off, len, nt, t0, t1, lane, acc); break;
    case 4: row_general<T, 4, U>(bal, as4, g0, off, len, nt, t0, t1, lane, acc); break;
    case 5: row_general<T, 5, U>(bal, as4, g0, off, len, nt, t0, t1, lane, acc); break;
    case 6: row_general<T, 6, U>(bal, as4, g0, off, len, nt, t0, t1, lane, acc); break;
    case 7: row_general<T, 7, U>(bal, as4, g0, off, len, nt, t0, t1, lane, acc); break;
    default: row_general<T, 8, U>(bal, as4, g0, off, len, nt, t0, t1, lane, acc); break;
  }
  return warp_sum(acc_total<2>(acc));
}

// ----------------------------------------------------------- main kernel --

// One CTA = one (row block, k-segment) pair: blockIdx.x = row_block * sg + s.
// Inside the CTA, warp w streams row slot w / sw over slice w % sw of the
// segment; slots advance by (W / sw) * R rows per pass.
template <class T, bool OUT_F32, int R, bool ALIGNED>
__global__ void __launch_bounds__(kMaxThreads, 2) gemv_rows_kernel(Params p) {
  constexpr int U = (R == 1) ? 8 : (R == 2 ? 4 : 2);
  extern __shared__ __align__(16) uint4 smem4[];
  uint4 *as4 = smem4;
  float *ps = reinterpret_cast<float *>(smem4 + (p.as_elems >> 3));

  const int W = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gs = blockIdx.x % p.sg;
  const int64_t rbk = blockIdx.x / p.sg;
  const int64_t q = p.n / p.nrb, rem = p.n % p.nrb;
  const int64_t r0 = rbk * q + (rbk < rem ? rbk : rem);
  const int64_t r1 = r0 + q + (rbk < rem ? 1 : 0);
  const int64_t j0 = (int64_t)gs * p.kseg;
  const int64_t len = (p.k - j0 < p.kseg) ? (p.k - j0) : p.kseg;

  allow_dependents();
  wait_for_predecessor();
  stage_a(p, as4, j0, len);
  __syncthreads();

  const int sw = p.sw, slots = W / sw, slot = warp / sw, s = warp % sw;
  const int64_t step = (int64_t)slots * R;
  for (int64_t base = r0; base < r1; base += step) {
    const int64_t i0 = base + (int64_t)slot * R;
    float v[R];
    if constexpr (ALIGNED) {
      const int nt = (int)(len >> 3);
      const int t0 = (int)((int64_t)nt * s / sw), t1 = (int)((int64_t)nt * (s + 1) / sw);
      if (i0 < r1) {  // warp-uniform; a slot past the CTA's rows reads nothing
        rows_aligned<T, R, U>(p, as4, i0, r1, j0, t0, t1, lane, v);
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = 0.f;
      }
    } else {
      v[0] = (i0 < r1) ? row_general_dispatch<T, U>(p, as4, i0, j0, len, s, sw, lane) : 0.f;
    }
    if (sw == 1) {
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (i0 + r < r1) store_out<T, OUT_F32>(p, gs, i0 + r, v[r]);
      }
    } else {
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) ps[(slot * R + r) * sw + s] = v[r];
      }
      __syncthreads();
      for (int t = threadIdx.x; t < slots * R; t += blockDim.x) {
        const int64_t row = base + t;
        if (row < r1) {
          float acc = 0.f;
          for (int s2 = 0; s2 < sw; ++s2) acc += ps[t * sw + s2];
          store_out<T, OUT_F32>(p, gs, row, acc);
        }
      }
      __syncthreads();
    }
  }
}

// Segments up to which the second pass of split-K gives each row one thread.
constexpr int kReduceRowThreads = 32;

// Second pass of split-K: c[row] = the sum over the sg segments of
// ws[s * n + row], rounded once to the output type.  Up to
// kReduceRowThreads segments, one thread adds a row's partials in segment
// order; beyond that (long rows split into many segments) a warp takes the
// row, lane l adding segments l, l + 32, ... in order, and the 32 lane sums
// are combined by the fixed xor-shuffle tree.  Either way the order is fixed
// for a given sg, so results are deterministic.
template <class T, bool OUT_F32>
__device__ __forceinline__ void store_reduced(void *c, int64_t row, float y) {
  if (OUT_F32) {
    static_cast<float *>(c)[row] = y;
  } else {
    static_cast<uint16_t *>(c)[row] = T::from_float(y);
  }
}

template <class T, bool OUT_F32>
__global__ void __launch_bounds__(256)
    gemv_splitk_reduce_kernel(const float *ws, void *c, int64_t n, int32_t sg, Epilogue ep) {
  allow_dependents();
  wait_for_predecessor();  // the partials come from the kernel before
  if (sg <= kReduceRowThreads) {
    for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < n;
         row += (int64_t)gridDim.x * blockDim.x) {
      float v = 0.f;
      for (int s = 0; s < sg; ++s) v += ws[(int64_t)s * n + row];
      store_reduced<T, OUT_F32>(c, row, apply_epilogue<T>(ep, row, v));
    }
  } else {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n; row += warps) {
      float v = 0.f;
      for (int s = lane; s < sg; s += 32) v += ws[(int64_t)s * n + row];
      v = warp_sum(v);
      if (lane == 0) store_reduced<T, OUT_F32>(c, row, apply_epilogue<T>(ep, row, v));
    }
  }
}

}  // namespace gemvk

// Explicit instantiation table for one input type (T = F16 or BF16).
#define GEMV_DEFINE_KERNEL_TABLE(T, SUFFIX)                                                    \
  namespace gemvk {                                                                             \
  MainKernel main_kernel_##SUFFIX(int out_f32, int variant, int R) {                           \
    if (variant == 1) {                                                                        \
      if (out_f32) {                                                                           \
        if (R == 1) return gemv_rows_kernel<T, true, 1, true>;                                 \
        if (R == 2) return gemv_rows_kernel<T, true, 2, true>;                                 \
        if (R == 4) return gemv_rows_kernel<T, true, 4, true>;                                 \
      } else {                                                                                 \
        if (R == 1) return gemv_rows_kernel<T, false, 1, true>;                                \
        if (R == 2) return gemv_rows_kernel<T, false, 2, true>;                                \
        if (R == 4) return gemv_rows_kernel<T, false, 4, true>;                                \
      }                                                                                        \
    } else if (variant == 2 && R == 1) {                                                       \
      return out_f32 ? gemv_rows_kernel<T, true, 1, false> : gemv_rows_kernel<T, false, 1, false>; \
    }                                                                                          \
    return nullptr;                                                                            \
  }                                                                                            \
  ReduceKernel reduce_kernel_##SUFFIX(int out_f32) {                                           \
    return out_f32 ? gemv_splitk_reduce_kernel<T, true> : gemv_splitk_reduce_kernel<T, false>; \
  }                                                                                            \
  }

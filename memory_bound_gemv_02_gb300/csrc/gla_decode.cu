// One decode step of gated linear attention on sm_103a (TileLang Case
// Studies, Case D "Background"):
//
//     S_new = diag(exp(gk)) @ S + outer(k, v),    o = scale * q^T @ S_new
//
// per head, S of shape (dk, dv) row-major.  The step reads the state once and
// writes it once -- bandwidth-bound like the GEMV -- and its output is a
// transposed matrix-vector product fused into the update.
//
// Design: a persistent grid walks the heads, G at a time per CTA round (G = 1
// for large heads; small heads side by side, so that each thread still has
// about four rows to stream).  For a round, exp(gk), k and q of its heads are
// staged in shared memory (fp32); the threads of head slot g own, thread t of
// the slot, the 16-byte column chunk t % (dv / VEC) of rows t / (dv / VEC),
// t / (dv / VEC) + RP, ... (so a warp's loads and stores cover contiguous
// rows: fully coalesced), update each element as fmaf(exp(gk_i), S_ij,
// k_i v_j) in fp32, store it rounded once, and accumulate q_i * S_new_ij
// (unrounded) for their columns.  The RP row partials of each column are
// added in shared memory in row-block order, so the result is deterministic.
// Four rows (large heads) or eight (small heads) are in flight per thread;
// the first batch is requested before the round's staging, so their
// latency overlaps it.  A pipelined form (gla_decode_pipe_kernel, the
// automatic choice where it applies) copies the next round into shared
// memory while the current one computes.
// S_new may be S itself (an in-place step): every element is read and then
// written by the same thread.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemv.h"
#include "gemv_kernels.cuh"

namespace gemvk {
namespace {

struct GlaParams {
  const void *q, *k, *v, *gk, *S;
  void *S_new, *o;
  int64_t bh;
  int32_t dk, dv;
  float scale;
  int32_t heads_per_cta;  // CTA layouts: heads processed side by side per round (G)
  int32_t early_state;    // GLA_PREFETCH_STATE: S is unwritten by the work in flight
};

struct F32 {};  // tag of the fp32 storage type

// Element access for the three storage types: VEC elements per 16 bytes.
template <class T>
struct GlaIo;

template <>
struct GlaIo<F16> {
  static constexpr int VEC = 8;
  static __device__ __forceinline__ float scalar(const void *p, int64_t i) {
    return F16::to_float(static_cast<const uint16_t *>(p)[i]);
  }
  static __device__ __forceinline__ void unpack(const uint4 &w, float (&f)[VEC]) { widen8<F16>(w, f); }
  static __device__ __forceinline__ uint4 pack(const float (&f)[VEC]) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = (uint32_t)F16::from_float(f[2 * q]) | ((uint32_t)F16::from_float(f[2 * q + 1]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  // As pack(), rounding each pair with one paired conversion (the same
  // nearest-even rounding of each element, hence the same bits).
  static __device__ __forceinline__ uint4 pack_pairs(const float (&f)[VEC]) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 h = __floats2half2_rn(f[2 * q], f[2 * q + 1]);
      w[q] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  // Elements i .. i + 3 (i % 4 == 0, p 8-byte aligned), by paired conversions.
  static __device__ __forceinline__ void store4(void *p, int64_t i, float a, float b, float c, float d) {
    const __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
    static_cast<uint2 *>(p)[i >> 2] =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
  }
};

template <>
struct GlaIo<BF16> {
  static constexpr int VEC = 8;
  static __device__ __forceinline__ float scalar(const void *p, int64_t i) {
    return BF16::to_float(static_cast<const uint16_t *>(p)[i]);
  }
  static __device__ __forceinline__ void unpack(const uint4 &w, float (&f)[VEC]) { widen8<BF16>(w, f); }
  static __device__ __forceinline__ uint4 pack(const float (&f)[VEC]) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = (uint32_t)BF16::from_float(f[2 * q]) | ((uint32_t)BF16::from_float(f[2 * q + 1]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  static __device__ __forceinline__ uint4 pack_pairs(const float (&f)[VEC]) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * q], f[2 * q + 1]);
      w[q] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  static __device__ __forceinline__ void store4(void *p, int64_t i, float a, float b, float c, float d) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    static_cast<uint2 *>(p)[i >> 2] =
        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
  }
};

template <>
struct GlaIo<F32> {
  static constexpr int VEC = 4;
  static __device__ __forceinline__ float scalar(const void *p, int64_t i) {
    return static_cast<const float *>(p)[i];
  }
  static __device__ __forceinline__ void unpack(const uint4 &w, float (&f)[VEC]) {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y); f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
  }
  static __device__ __forceinline__ uint4 pack(const float (&f)[VEC]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  static __device__ __forceinline__ uint4 pack_pairs(const float (&f)[VEC]) { return pack(f); }
  static __device__ __forceinline__ void store4(void *p, int64_t i, float a, float b, float c, float d) {
    static_cast<float4 *>(p)[i >> 2] = make_float4(a, b, c, d);
  }
};

constexpr int kGlaThreads = 256;
constexpr int kGlaMaxDk = 4096;
// Rows of 16-byte chunks in flight per thread in the CTA layout: 8 for heads
// of at most kGlaSmallHeadChunks chunks (with registers capped for 3 CTAs
// per SM: 96 KB in flight per SM), 4 for larger heads (4 CTAs per SM).
// Measured on GB300 back to back: 64 x 64 heads 7-9 % faster with 8, 128 x
// 128 and 256 x 256 heads 3-8 % slower.
constexpr int kGlaRowsInFlight = 4;
constexpr int kGlaRowsInFlightSmall = 8;
constexpr int64_t kGlaSmallHeadChunks = 1024;

// Floats to add after x floats to reach a multiple of 4 (16 bytes).
__host__ __device__ constexpr int gla_pad4(int64_t x) { return (int)((4 - (x & 3)) & 3); }

// 16-byte store of data written once (no L1 allocation needed).
__device__ __forceinline__ void stg_stream(uint4 *p, const uint4 &v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// o of a round of nh heads from the row-block partials part[G][RP][dv]:
// o[h0 * dv + x] = scale * (0 + part[g][0][j] + part[g][1][j] + ...), x =
// g * dv + j, the row blocks added in ascending order.  Each thread takes
// four consecutive outputs (one 16-byte read of the partials per row block,
// one store of the four results through paired conversions: the same
// rounding, hence the same bits as one at a time); o is 16-byte aligned (the
// host checks it) and dv % 4 == 0, so each store is aligned.  At 16384 x 16
// x 64 fp16 a round has 1024 outputs, and storing them one at a time took
// 21 % more instructions than a 64 x 64 step of the same bytes.
template <class T>
__device__ __forceinline__ void store_o(const GlaParams &p, const float *part, int64_t h0, int nh, int dv, int RP,
                                        int t, int nthreads) {
  using IO = GlaIo<T>;
  const int n4 = nh * dv / 4;  // dv % 4 == 0 (dv % VEC == 0)
  for (int x4 = t; x4 < n4; x4 += nthreads) {
    const int x = 4 * x4, g = x / dv, j = x % dv;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int rb = 0; rb < RP; ++rb) {
      const float4 v = *reinterpret_cast<const float4 *>(part + (g * RP + rb) * dv + j);
      s0 += v.x;
      s1 += v.y;
      s2 += v.z;
      s3 += v.w;
    }
    IO::store4(p.o, h0 * dv + x, p.scale * s0, p.scale * s1, p.scale * s2, p.scale * s3);
  }
}

// Store a thread's VEC partial sums of o at float offset `off` of `part`
// (a multiple of 4) as 16-byte vectors.  With 8 per thread, neighbouring
// lanes' offsets are 8 floats apart and lanes 4 apart would hit the same
// bank group; those with bit 5 of the offset set store their second half
// first, so that each group of 8 lanes writes 8 distinct bank groups.
template <int VEC>
__device__ __forceinline__ void store_partials(float *part, int off, const float (&acc)[VEC]) {
  float4 *d = reinterpret_cast<float4 *>(part + off);
  if constexpr (VEC == 4) {
    d[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  } else {
    static_assert(VEC == 8, "16-byte chunks hold 4 or 8 elements");
    const float4 lo = make_float4(acc[0], acc[1], acc[2], acc[3]);
    const float4 hi = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if ((off >> 5) & 1) {
      d[1] = hi;
      d[0] = lo;
    } else {
      d[0] = lo;
      d[1] = hi;
    }
  }
}

// Ask L2 for bytes [p, p + min(bytes, 32 * 16 KB)), a multiple of 16, in
// pieces of at most 16 KB, piece i by lane i of the calling warp.  Issued
// before waiting on the preceding kernel: a prefetch reads nothing into the
// kernel, and L2 is where that kernel's writes land, so it needs no promise.
constexpr int64_t kGlaL2Piece = 16 * 1024;
__device__ __forceinline__ void prefetch_l2_pieces(const void *p, int64_t bytes, int lane) {
  const int64_t off = (int64_t)lane * kGlaL2Piece;
  if (off < bytes) {
    const int64_t nb = bytes - off < kGlaL2Piece ? bytes - off : kGlaL2Piece;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char *>(p) + off),
                 "r"((uint32_t)nb)
                 : "memory");
  }
}

// The state bytes of round r's heads (at most 64 KB from the round's start),
// for the pipelined layout's first round.
__device__ __forceinline__ void prefetch_first_round(const GlaParams &p, int es, int64_t r, int G) {
  const int64_t h0 = r * G;
  const int64_t nh = p.bh - h0 < G ? p.bh - h0 : G;
  const int64_t hb = (int64_t)p.dk * p.dv * es;
  const int64_t bytes = nh * hb < 4 * kGlaL2Piece ? nh * hb : 4 * kGlaL2Piece;
  prefetch_l2_pieces(static_cast<const char *>(p.S) + h0 * hb, bytes, threadIdx.x & 31);
}

template <class T, int RIF>
__device__ __forceinline__ void gla_decode_body(const GlaParams &p) {
  using IO = GlaIo<T>;
  constexpr int VEC = IO::VEC;
  extern __shared__ __align__(16) float gsm[];
  const int dk = p.dk, dv = p.dv, G = p.heads_per_cta;
  const int cpr = dv / VEC;               // 16-byte chunks per row
  const int TPG = kGlaThreads / G;        // threads per head
  const int RP = TPG / cpr;               // row blocks per head (>= 1: the host keeps G * cpr <= kGlaThreads)
  float *dec = gsm;                       // exp(gk)   [G][dk]
  float *kk = dec + G * dk;               // k         [G][dk]
  float *qq = kk + G * dk;                // q         [G][dk]
  float *part = qq + G * dk + gla_pad4(3 * G * dk);  // row-block partials of o [G][RP][dv], 16-byte aligned
  const int t = threadIdx.x;
  const int gi = t / TPG, tl = t % TPG;   // head slot of this thread, its index in the slot
  // Launched as a programmatic dependent launch: let the next kernel be
  // scheduled early, and touch no memory before the previous one is done --
  // except, with GLA_PREFETCH_STATE, the first state rows of the first
  // round, which the caller promised no work in flight writes.  (An L2
  // prefetch of them before the wait, as the pipelined layout makes,
  // measured 1-8 % slower here.)
  allow_dependents();
  const int64_t rounds = (p.bh + G - 1) / G;
  bool waited = p.early_state == 0;
  if (waited) wait_for_predecessor();
  const int cc = tl % cpr, rl = tl / cpr;

  for (int64_t r = blockIdx.x; r < rounds; r += gridDim.x) {
    const int64_t h0 = r * G;                    // first head of this round
    const int nh = (p.bh - h0 < G) ? (int)(p.bh - h0) : G;
    const int64_t h = h0 + gi;                   // this thread's head
    const bool active = rl < RP && gi < nh;
    const uint4 *Srow = reinterpret_cast<const uint4 *>(p.S) + (h * dk) * (int64_t)cpr + cc;
    // The first rows of the head are requested before q, k, gk are staged,
    // so that the two latencies overlap.
    uint4 sv[RIF];
#pragma unroll
    for (int u = 0; u < RIF; ++u) {
      const int i = rl + u * RP;
      sv[u] = (active && i < dk) ? ldg_stream(Srow + (int64_t)i * cpr) : zero4();
    }
    if (!waited) {
      wait_for_predecessor();
      waited = true;
    }
    for (int x = t; x < nh * dk; x += kGlaThreads) {
      dec[x] = expf(IO::scalar(p.gk, h0 * dk + x));
      kk[x] = IO::scalar(p.k, h0 * dk + x);
      qq[x] = IO::scalar(p.q, h0 * dk + x);
    }
    __syncthreads();
    if (active) {
      const float *hd = dec + gi * dk, *hk = kk + gi * dk, *hq = qq + gi * dk;
      // this thread's VEC elements of v (16-byte aligned: dv % VEC == 0)
      float vv[VEC];
      IO::unpack(__ldg(reinterpret_cast<const uint4 *>(p.v) + (h * dv) / VEC + cc), vv);
      float acc[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
      uint4 *Nrow = reinterpret_cast<uint4 *>(p.S_new) + (h * dk) * (int64_t)cpr + cc;
      for (int i0 = rl; i0 < dk; i0 += RP * RIF) {
        if (i0 != rl) {
#pragma unroll
          for (int u = 0; u < RIF; ++u) {
            const int i = i0 + u * RP;
            sv[u] = (i < dk) ? ldg_stream(Srow + (int64_t)i * cpr) : zero4();
          }
        }
#pragma unroll
        for (int u = 0; u < RIF; ++u) {
          const int i = i0 + u * RP;
          if (i < dk) {
            float s[VEC], sn[VEC];
            IO::unpack(sv[u], s);
            const float di = hd[i], ki = hk[i], qi = hq[i];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              sn[e] = fmaf(di, s[e], ki * vv[e]);
              acc[e] = fmaf(qi, sn[e], acc[e]);
            }
            // paired conversions (same bits): 1024 x 256 x 256 bf16 45.24 ->
            // 44.65 us back to back on GB300, fp16 45.22 -> 44.66
            stg_stream(Nrow + (int64_t)i * cpr, IO::pack_pairs(sn));
          }
        }
      }
      store_partials<VEC>(part, (gi * RP + rl) * dv + cc * VEC, acc);
    }
    __syncthreads();
    store_o<T>(p, part, h0, nh, dv, RP, t, kGlaThreads);
    __syncthreads();  // dec/kk/qq/part are reused by the next round
  }
}

// The CTA layout for large heads (4 rows in flight, 4 CTAs of 64 registers
// per SM) and for small heads (8 rows in flight, registers capped for 3 CTAs
// per SM).
template <class T>
__global__ void __launch_bounds__(kGlaThreads) gla_decode_kernel(GlaParams p) {
  gla_decode_body<T, kGlaRowsInFlight>(p);
}

template <class T>
__global__ void __launch_bounds__(kGlaThreads, 3) gla_decode_kernel_small(GlaParams p) {
  gla_decode_body<T, kGlaRowsInFlightSmall>(p);
}

// ---------------------------------------------------------------- pipelined
// The CTA layout with the next round staged by asynchronous copies
// (cp.async, 16 bytes each) into a second shared-memory buffer while the
// current round computes, so that a CTA's loads never wait for its round
// barriers.  For rounds of at most kGlaPipeRoundChunks 16-byte state chunks
// with q, k, gk and v rows that are whole 16-byte chunks.
//
// Shared memory, per buffer b in {0, 1}: the round's state, as in global
// memory ([G][dk][cpr] chunks: each thread copies exactly the chunks it will
// read, so its own wait makes them visible), then q, k, gk ([G][dk] each,
// QC chunks apart) and v ([G][dv]) in the input type, copied by all threads
// and read by all after a barrier; then o's row-block partials [G][RP][dv]
// and the round's exp(gk), k and q as fp32 ([G][dk] each, written by all
// threads after that barrier and read after a second one).
// The thread mapping, the fmaf per element and the order of every sum are
// those of gla_decode_kernel with the same G: S_new is bit-identical, and o
// too where the two choose the same G (G sets the row blocks o is summed in).
// Before waiting on the preceding kernel, warp 0 asks L2 for the first
// round's state (or, with GLA_PREFETCH_STATE, every thread already copies
// its part of it): measured 3-8 % faster back to back.  A round's q, k, gk
// and v are copied before its state (the whole round waits for both, and
// the small rows no longer queue behind the state's chunks): 4096 x 64 x
// 64 fp16 12.60 -> 12.21 us back to back, 16384 x 16 x 64 15.41 -> 15.02,
// 2048 x 128 x 128 bf16 21.95 -> 21.79, 4096 x 128 x 128 bf16 42.04 ->
// 42.23.  (Loading the CTA layout's first q, k, gk values ahead of its
// state rows instead measured up to 12 % slower there.)
constexpr int kGlaPipeRoundChunks = 2048;
constexpr int64_t kGlaPairPackMaxHead = 16 * 1024;  // state bytes of a head up to which S_new is stored through pack_pairs
// Shared memory of one CTA at most: two CTAs per SM (228 KB, 1 KB reserved
// per CTA).  More heads per round measured faster than more CTAs per SM:
// 4096 x 64 x 64 fp16 13.8 us with 4 heads per round and 2 CTAs per SM
// against 15.0 us with 2 heads and 4 CTAs; one CTA per SM with rounds of
// up to 4096 chunks was slower on every workload (16.1 us here).
constexpr int64_t kGlaPipeMaxSmem = 110 * 1024;

// Dynamic shared memory of the pipelined layout: two buffers of a round's
// state, q, k, gk and v (16-byte chunks), then o's row-block partials, then
// the round's exp(gk), k and q in fp32.
int64_t gla_pipe_smem(int G, int64_t dk, int64_t dv, int cpr, int es) {
  const int RP = (kGlaThreads / G) / cpr;
  const int64_t buf = (int64_t)G * dk * cpr + 3 * ((int64_t)G * dk * es / 16) + (int64_t)G * cpr;
  return 2 * buf * 16 + (int64_t)G * RP * dv * (int64_t)sizeof(float) + 3 * (int64_t)G * dk * (int64_t)sizeof(float);
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most one committed group of this thread is still pending.
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// PAIRS: store S_new through IO::pack_pairs (same bits).  Measured on GB300
// back to back, it is faster for heads of at most kGlaPairPackMaxHead bytes
// (4096 x 64 x 64 fp16 13.71 -> 12.59 us, 16384 x 16 x 64 fp16 16.51 ->
// 15.47, 8192 x 64 x 64 bf16 22.50 -> 22.36) and slower for some larger ones
// (4096 x 128 x 128 fp16 42.55 -> 44.00, bf16 42.08 -> 43.90).
template <class T, bool PAIRS>
__global__ void __launch_bounds__(kGlaThreads) gla_decode_pipe_kernel(GlaParams p) {
  using IO = GlaIo<T>;
  constexpr int VEC = IO::VEC;
  constexpr int ES = 16 / VEC;  // element size in bytes
  extern __shared__ uint4 gsm4[];
  const int dk = p.dk, dv = p.dv, G = p.heads_per_cta;
  const int cpr = dv / VEC;
  const int TPG = kGlaThreads / G, RP = TPG / cpr;
  const int SC = G * dk * cpr;        // state chunks per buffer
  const int QC = G * dk * ES / 16;    // chunks of one of q, k, gk per buffer (dk * ES % 16 == 0)
  const int BUF = SC + 3 * QC + G * cpr;
  float *part = reinterpret_cast<float *>(gsm4 + 2 * BUF);
  float *dec = part + G * RP * dv, *kk = dec + G * dk, *qq = kk + G * dk;  // [G][dk] fp32 each
  const int t = threadIdx.x;
  const int gi = t / TPG, tl = t % TPG;
  const int cc = tl % cpr, rl = tl / cpr;
  const int64_t rounds = (p.bh + G - 1) / G;
  const uint4 *Sg = reinterpret_cast<const uint4 *>(p.S);

  // This thread's state chunks of round r into buffer b.
  auto issue_state = [&](int64_t r, int b) {
    const int64_t h0 = r * G;
    const int nh = (p.bh - h0 < G) ? (int)(p.bh - h0) : G;
    if (rl < RP && gi < nh) {
      uint4 *dst = gsm4 + (size_t)b * BUF + (size_t)gi * dk * cpr + cc;
      const uint4 *src = Sg + ((h0 + gi) * dk) * (int64_t)cpr + cc;
      for (int i = rl; i < dk; i += RP) cp_async16(dst + (size_t)i * cpr, src + (int64_t)i * cpr);
    }
  };
  // Round r's q, k, gk and v into buffer b, dealt over all threads.
  auto issue_vectors = [&](int64_t r, int b) {
    const int64_t h0 = r * G;
    const int nh = (p.bh - h0 < G) ? (int)(p.bh - h0) : G;
    const int nq = nh * dk * ES / 16, nv = nh * cpr;
    uint4 *base = gsm4 + (size_t)b * BUF + SC;
    const int64_t q0 = h0 * dk * ES / 16;
    for (int x = t; x < 3 * nq + nv; x += kGlaThreads) {
      if (x < 3 * nq) {
        const int a = x / nq, y = x % nq;
        const void *v = a == 0 ? p.q : a == 1 ? p.k : p.gk;
        cp_async16(base + a * QC + y, reinterpret_cast<const uint4 *>(v) + q0 + y);
      } else {
        const int y = x - 3 * nq;
        cp_async16(base + 3 * QC + y, reinterpret_cast<const uint4 *>(p.v) + h0 * cpr + y);
      }
    }
  };

  allow_dependents();
  int64_t r = blockIdx.x;
  if (r >= rounds) {
    wait_for_predecessor();
    return;
  }
  // Launched as a programmatic dependent launch: with GLA_PREFETCH_STATE the
  // first round's state is requested before waiting for the preceding
  // kernel; without it, warp 0 only asks L2 for it.
  if (p.early_state) {
    issue_state(r, 0);
    wait_for_predecessor();
  } else {
    if (t < 32) prefetch_first_round(p, ES, r, G);
    wait_for_predecessor();
    issue_vectors(r, 0);
    issue_state(r, 0);
  }
  if (p.early_state) issue_vectors(r, 0);
  cp_async_commit();
  for (int b = 0; r < rounds; r += gridDim.x, b ^= 1) {
    const int64_t rn = r + gridDim.x;
    if (rn < rounds) {  // buffer b ^ 1 was last read before the previous round's second barrier
      issue_vectors(rn, b ^ 1);
      issue_state(rn, b ^ 1);
    }
    cp_async_commit();
    cp_async_wait_all_but_one();  // this thread's copies of round r have landed
    __syncthreads();              // and everyone's (q, k, gk, v are shared)
    const int64_t h0 = r * G;
    const int nh = (p.bh - h0 < G) ? (int)(p.bh - h0) : G;
    // The round's per-row factors, once each in fp32: the cpr threads that
    // share a row would otherwise each evaluate its exp(gk) (measured on
    // GB300 back to back: 2048 x 128 x 128 bf16 22.9 -> 21.9 us, 4096 x 128 x
    // 128 bf16 44.6 -> 42.1 us, small heads 0.1-0.8 % faster; same values).
    {
      const uint4 *buf = gsm4 + (size_t)b * BUF;
      const void *qs = buf + SC, *ks = buf + SC + QC, *gs = buf + SC + 2 * QC;
      for (int x = t; x < nh * dk; x += kGlaThreads) {
        dec[x] = expf(IO::scalar(gs, x));
        kk[x] = IO::scalar(ks, x);
        qq[x] = IO::scalar(qs, x);
      }
    }
    __syncthreads();
    if (rl < RP && gi < nh) {
      const int64_t h = h0 + gi;
      const uint4 *buf = gsm4 + (size_t)b * BUF;
      const uint4 *st = buf + (size_t)gi * dk * cpr + cc;
      float vv[VEC], acc[VEC];
      IO::unpack(buf[SC + 3 * QC + gi * cpr + cc], vv);
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
      uint4 *Nrow = reinterpret_cast<uint4 *>(p.S_new) + (h * dk) * (int64_t)cpr + cc;
      for (int i = rl; i < dk; i += RP) {
        float s[VEC], sn[VEC];
        IO::unpack(st[(size_t)i * cpr], s);
        const int x = gi * dk + i;
        const float di = dec[x], ki = kk[x], qi = qq[x];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          sn[e] = fmaf(di, s[e], ki * vv[e]);
          acc[e] = fmaf(qi, sn[e], acc[e]);
        }
        stg_stream(Nrow + (int64_t)i * cpr, PAIRS ? IO::pack_pairs(sn) : IO::pack(sn));
      }
      store_partials<VEC>(part, (gi * RP + rl) * dv + cc * VEC, acc);
    }
    __syncthreads();
    store_o<T>(p, part, h0, nh, dv, RP, t, kGlaThreads);
  }
}

// One warp per head, for many small heads (dv * element size <= 512 bytes):
// lane l owns 16-byte column chunk l % cpr of rows l / cpr, l / cpr + RPW,
// ... (RPW = 32 / cpr row groups per warp), with 8 of its rows in flight,
// their exp(gk_i), k_i, q_i loaded beside them.  No block barrier: o's
// column sums are reduced over the RPW row groups by shuffles, in row-group
// order (deterministic).  The update of each element is the same fmaf as in
// gla_decode_kernel, so S_new is bit-identical between the two layouts.
constexpr int kGlaWarpRows = 8;

template <class T>
__global__ void __launch_bounds__(kGlaThreads) gla_decode_warp_kernel(GlaParams p) {
  using IO = GlaIo<T>;
  constexpr int VEC = IO::VEC;
  constexpr int RW = kGlaWarpRows;
  const int dk = p.dk, dv = p.dv;
  const int cpr = dv / VEC;  // <= 32 (host)
  const int RPW = 32 / cpr;
  const int lane = threadIdx.x & 31;
  const int cc = lane % cpr, rw = lane / cpr;
  const bool active = rw < RPW;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  allow_dependents();
  wait_for_predecessor();
  for (int64_t h = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); h < p.bh; h += nw) {
    float vv[VEC], acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = vv[e] = 0.f;
    if (active) IO::unpack(__ldg(reinterpret_cast<const uint4 *>(p.v) + h * cpr + cc), vv);
    const uint4 *Srow = reinterpret_cast<const uint4 *>(p.S) + (h * dk) * (int64_t)cpr + cc;
    uint4 *Nrow = reinterpret_cast<uint4 *>(p.S_new) + (h * dk) * (int64_t)cpr + cc;
    for (int i0 = rw; i0 < dk; i0 += RPW * RW) {
      uint4 sv[RW];
      float gv[RW], kv[RW], qv[RW];
#pragma unroll
      for (int u = 0; u < RW; ++u) {
        const int i = i0 + u * RPW;
        const bool ok = active && i < dk;
        sv[u] = ok ? ldg_stream(Srow + (int64_t)i * cpr) : zero4();
        gv[u] = ok ? IO::scalar(p.gk, h * dk + i) : 0.f;
        kv[u] = ok ? IO::scalar(p.k, h * dk + i) : 0.f;
        qv[u] = ok ? IO::scalar(p.q, h * dk + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < RW; ++u) {
        const int i = i0 + u * RPW;
        if (active && i < dk) {
          float s[VEC], sn[VEC];
          IO::unpack(sv[u], s);
          const float di = expf(gv[u]);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            sn[e] = fmaf(di, s[e], kv[u] * vv[e]);
            acc[e] = fmaf(qv[u], sn[e], acc[e]);
          }
          stg_stream(Nrow + (int64_t)i * cpr, IO::pack(sn));
        }
      }
    }
    float tot[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      tot[e] = 0.f;
      for (int r = 0; r < RPW; ++r) tot[e] += __shfl_sync(0xffffffffu, acc[e], cc + r * cpr);
      tot[e] *= p.scale;
    }
    if (rw == 0) stg_stream(reinterpret_cast<uint4 *>(p.o) + h * cpr + cc, IO::pack(tot));
  }
}

// Launch a GLA kernel as a programmatic dependent launch (the kernels wait
// for the preceding kernel before touching memory, so this orders like a
// plain launch and only lets the launch overlap the predecessor's drain).
cudaError_t pdl_launch(const void *fn, unsigned grid, size_t smem, cudaStream_t stream, GlaParams p) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kGlaThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  lc.attrs = attr;
  lc.numAttrs = 1;
  void *args[] = {&p};
  cudaError_t e = cudaLaunchKernelExC(&lc, fn, args);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

// Grid for `units` rounds of work dealt round-robin over at most `cap`
// resident CTAs.  The fewest rounds per CTA the cap allows, then the fewest
// CTAs that still finish in that many rounds, so that no CTA starts a last
// round that most others skip (2048 heads over 608 slots: 512 CTAs of 4
// rounds, not 608 CTAs of which 224 run a fourth) -- unless that drops more
// than a fifth of the cap: each CTA round is latency-bound, and fewer CTAs
// then cost more bandwidth than the ragged last round (measured on GB300 back
// to back: 1-3 % faster at 84-96 % of the cap, 1-3 % slower at 75 %).
int64_t balanced_grid(int64_t units, int64_t cap) {
  if (units <= cap) return units;
  const int64_t per = (units + cap - 1) / cap;
  const int64_t grid = (units + per - 1) / per;
  return 5 * grid >= 4 * cap ? grid : cap;
}

bool overlap_bytes(const void *p, int64_t pb, const void *q, int64_t qb) {
  const uintptr_t a0 = (uintptr_t)p, a1 = a0 + (uintptr_t)pb;
  const uintptr_t b0 = (uintptr_t)q, b1 = b0 + (uintptr_t)qb;
  return a0 < b1 && b0 < a1;
}

}  // namespace
}  // namespace gemvk

using namespace gemvk;

extern "C" int gla_decode_ex(const void *q, const void *k, const void *v, const void *gk, const void *S,
                             void *S_new, void *o, int64_t bh, int64_t dk, int64_t dv, float scale, int dtype,
                             int variant, int flags, cudaStream_t stream) {
  if (dtype != GLA_F16 && dtype != GLA_BF16 && dtype != GLA_F32) return GEMV_ERR_DTYPE;
  if (flags & ~GLA_PREFETCH_STATE) return GEMV_ERR_ARG;
  if (variant < GLA_VARIANT_AUTO || variant > GLA_VARIANT_PIPE) return GEMV_ERR_CONFIG;
  if (bh < 0 || dk < 0 || dv < 0 || dk > kGlaMaxDk) return GEMV_ERR_ARG;
  if (bh == 0 || dv == 0) return GEMV_OK;
  const int es = dtype == GLA_F32 ? 4 : 2;
  const int VEC = 16 / es;
  if (dv % VEC != 0 || dv / VEC > kGlaThreads) return GEMV_ERR_ARG;
  if (o == nullptr || v == nullptr) return GEMV_ERR_ARG;
  if (dk > 0 && (q == nullptr || k == nullptr || gk == nullptr || S == nullptr || S_new == nullptr))
    return GEMV_ERR_ARG;
  if (((uintptr_t)v | (uintptr_t)o) & 15u) return GEMV_ERR_ALIGN;
  if (dk > 0 && (((uintptr_t)S | (uintptr_t)S_new) & 15u)) return GEMV_ERR_ALIGN;
  if (dk > 0 && (((uintptr_t)q | (uintptr_t)k | (uintptr_t)gk) % (uintptr_t)es)) return GEMV_ERR_ALIGN;
  const int64_t sbytes = bh * dk * dv * es, obytes = bh * dv * es, vecbytes = bh * dk * es;
  // S_new may be S itself (in place), but must not partly overlap it; o
  // overlaps nothing.
  if (dk > 0 && S_new != S && overlap_bytes(S_new, sbytes, S, sbytes)) return GEMV_ERR_ALIAS;
  if (overlap_bytes(o, obytes, v, obytes)) return GEMV_ERR_ALIAS;
  if (dk > 0 && (overlap_bytes(o, obytes, S, sbytes) || overlap_bytes(o, obytes, S_new, sbytes) ||
                 overlap_bytes(o, obytes, q, vecbytes) || overlap_bytes(o, obytes, k, vecbytes) ||
                 overlap_bytes(o, obytes, gk, vecbytes)))
    return GEMV_ERR_ALIAS;
  if (dk > 0 && (overlap_bytes(S_new, sbytes, q, vecbytes) || overlap_bytes(S_new, sbytes, k, vecbytes) ||
                 overlap_bytes(S_new, sbytes, gk, vecbytes) || overlap_bytes(S_new, sbytes, v, obytes)))
    return GEMV_ERR_ALIAS;

  int dev = -1, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMV_ERR_DEVICE;
  }
  if (major != 10 || minor != 3) return GEMV_ERR_DEVICE;
  if (!on_device(dev, {dk > 0 ? q : nullptr, dk > 0 ? k : nullptr, v, dk > 0 ? gk : nullptr,
                       dk > 0 ? S : nullptr, dk > 0 ? S_new : nullptr, o}))
    return GEMV_ERR_DEVICE;
  const int cpr = (int)(dv / VEC);
  // The pipelined CTA layout needs q, k, gk rows of whole 16-byte chunks and
  // a round (G heads, G >= 1) of at most kGlaPipeRoundChunks state chunks.
  const bool pipe_ok = dk > 0 && (dk * es) % 16 == 0 && ((((uintptr_t)q | (uintptr_t)k | (uintptr_t)gk) & 15u) == 0) &&
                       dk * cpr <= kGlaPipeRoundChunks && gla_pipe_smem(1, dk, dv, cpr, es) <= kGlaPipeMaxSmem;
  // The CTA layout with several heads per round measured faster than a
  // warp per head on every workload tried (4096 x 64 x 64 fp16: 16.0 vs
  // 18.2 us; 16384 x 16 x 64 fp16: 19.0 vs 27.0 us; 4096 x 128 x 128 bf16:
  // 45.4 vs 53.6 us), and its pipelined form faster still on every
  // workload it takes (2048 x 128 x 128 bf16: 23.1 vs 25.8 us; 8192 x 64 x
  // 64 bf16: 24.6 vs 27.5 us; 16384 x 16 x 64 fp16: 16.7 vs 19.0 us).
  if (variant == GLA_VARIANT_AUTO) variant = pipe_ok ? GLA_VARIANT_PIPE : GLA_VARIANT_CTA;
  if (variant == GLA_VARIANT_WARP && cpr > 32) return GEMV_ERR_CONFIG;
  if (variant == GLA_VARIANT_PIPE && !pipe_ok) return GEMV_ERR_CONFIG;
  GlaParams p;
  p.q = q; p.k = k; p.v = v; p.gk = gk; p.S = S; p.S_new = S_new; p.o = o;
  p.bh = bh; p.dk = (int32_t)dk; p.dv = (int32_t)dv; p.scale = scale; p.heads_per_cta = 1;
  p.early_state = (flags & GLA_PREFETCH_STATE) ? 1 : 0;
  if (variant == GLA_VARIANT_WARP) {
    void (*fw)(GlaParams) = dtype == GLA_F16 ? gla_decode_warp_kernel<F16>
                            : dtype == GLA_BF16 ? gla_decode_warp_kernel<BF16> : gla_decode_warp_kernel<F32>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void *)fw, kGlaThreads, 0) != cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      return GEMV_ERR_CONFIG;
    }
    const int64_t warps = kGlaThreads / 32;
    const int64_t grid = (balanced_grid(bh, (int64_t)sms * per_sm * warps) + warps - 1) / warps;
    if (pdl_launch((const void *)fw, (unsigned)grid, 0, stream, p) != cudaSuccess) return GEMV_ERR_CUDA;
    return GEMV_OK;
  }
  if (variant == GLA_VARIANT_PIPE) {
    // Heads per round: as many as keep a round within kGlaPipeRoundChunks
    // chunks, the buffers within kGlaPipeMaxSmem, and at least one row block
    // of cpr threads per head.
    int G = 1;
    while (2 * G * cpr <= kGlaThreads && (int64_t)2 * G <= bh && (int64_t)dk * cpr * (2 * G) <= kGlaPipeRoundChunks &&
           gla_pipe_smem(2 * G, dk, dv, cpr, es) <= kGlaPipeMaxSmem)
      G *= 2;
    p.heads_per_cta = G;
    const size_t smem = (size_t)gla_pipe_smem(G, dk, dv, cpr, es);
    const bool pairs = dk * dv * es <= kGlaPairPackMaxHead;
    void (*fn)(GlaParams) = dtype == GLA_F16    ? (pairs ? gla_decode_pipe_kernel<F16, true> : gla_decode_pipe_kernel<F16, false>)
                            : dtype == GLA_BF16 ? (pairs ? gla_decode_pipe_kernel<BF16, true> : gla_decode_pipe_kernel<BF16, false>)
                                                : gla_decode_pipe_kernel<F32, false>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute((const void *)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return GEMV_ERR_CUDA;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void *)fn, kGlaThreads, smem) != cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      return GEMV_ERR_CONFIG;
    }
    const int64_t grid = balanced_grid((bh + G - 1) / G, (int64_t)sms * per_sm);
    if (pdl_launch((const void *)fn, (unsigned)grid, smem, stream, p) != cudaSuccess) return GEMV_ERR_CUDA;
    return GEMV_OK;
  }
  // Rows in flight per thread, and heads side by side per CTA round: enough
  // that each thread has about RIF rows of its head to stream (small
  // heads), at least one row block of cpr threads per head.
  const bool small = (int64_t)dk * cpr <= kGlaSmallHeadChunks;
  const int RIF = small ? kGlaRowsInFlightSmall : kGlaRowsInFlight;
  int G = 1;
  while (2 * G * cpr <= kGlaThreads && (int64_t)2 * G <= bh &&
         (int64_t)dk * cpr * (2 * G) <= (int64_t)RIF * kGlaThreads)
    G *= 2;
  p.heads_per_cta = G;
  const int RP = (kGlaThreads / G) / cpr;
  const size_t smem = (size_t)(3 * (int64_t)G * dk + gla_pad4(3 * (int64_t)G * dk) + (int64_t)G * RP * dv) *
                      sizeof(float);
  void (*fn)(GlaParams);
  if (small) {
    fn = dtype == GLA_F16 ? gla_decode_kernel_small<F16>
         : dtype == GLA_BF16 ? gla_decode_kernel_small<BF16> : gla_decode_kernel_small<F32>;
  } else {
    fn = dtype == GLA_F16 ? gla_decode_kernel<F16> : dtype == GLA_BF16 ? gla_decode_kernel<BF16> : gla_decode_kernel<F32>;
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute((const void *)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return GEMV_ERR_CUDA;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void *)fn, kGlaThreads, smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    return GEMV_ERR_CONFIG;
  }
  const int64_t grid = balanced_grid((bh + G - 1) / G, (int64_t)sms * per_sm);
  if (pdl_launch((const void *)fn, (unsigned)grid, smem, stream, p) != cudaSuccess) return GEMV_ERR_CUDA;
  return GEMV_OK;
}

extern "C" int gla_decode(const void *q, const void *k, const void *v, const void *gk, const void *S, void *S_new,
                          void *o, int64_t bh, int64_t dk, int64_t dv, float scale, int dtype, cudaStream_t stream) {
  return gla_decode_ex(q, k, v, gk, S, S_new, o, bh, dk, dv, scale, dtype, GLA_VARIANT_AUTO, 0, stream);
}

// Internal declarations shared by the host API and the kernel translation
// units of the GEMV library.  Not installed; the public surface is gemv.h.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#include <initializer_list>

#ifdef __CUDACC__
#define GEMV_HD __host__ __device__
#else
#define GEMV_HD
#endif

namespace gemvk {

// Fused epilogue applied to each row total before the single rounding:
// y = act(alpha * acc + beta * bias[row]) (bias optional, in the input type
// or fp32).  alpha = 1, no bias and act = 0 leave acc unchanged.
struct Epilogue {
  float alpha;
  float beta;
  const void *bias;  // n elements or nullptr
  int32_t bias_f32;  // 1: bias is fp32, 0: bias has the input type
  int32_t act;       // 0 none, 1 relu, 2 sigmoid, 3 silu
};

// Launch parameters of the main streaming kernel (passed by value).
struct Params {
  const uint16_t *B;  // n x k row-major, element (2-byte) aligned
  const uint16_t *a;  // k elements
  void *c;            // output, when grid_split == 1
  float *ws;          // fp32 partials ws[s * n + row], when grid_split > 1
  int64_t n;
  int64_t k;
  int64_t ldb;        // row stride of B in elements (>= k)
  int64_t kseg;       // columns per k-segment
  int32_t base_off;   // (address of B / 2) mod 8: B's element offset within a 16-byte block
  int32_t sg;         // grid split (CTAs per row block)
  int32_t sw;         // warp split (warps per row inside a CTA)
  int32_t nrb;        // row blocks = gridDim.x / sg
  int32_t as_elems;   // staged a elements per CTA (multiple of 8, >= kseg + 24)
  int32_t flags;      // kFlag* bits | (L2 prefetch rounds << kFlagL2Shift)
  Epilogue ep;
  // Tiles kernel: sw = S (warps per row, slices), nrb = C (CTAs per k-segment).
  // Bulk kernel only:
  int32_t stages;      // ring buffers per warp
  int32_t wait_polls;  // mbarrier polls per ring wait before giving up
  uint32_t *timeouts;  // per-device counter of ring waits that gave up
};

typedef void (*MainKernel)(Params);
typedef void (*ReduceKernel)(const float *, void *, int64_t, int32_t, Epilogue);

// Kernel lookup.  in16: 0 fp16, 1 bf16.  out_f32: 0 same as input, 1 fp32.
// variant: 1 aligned rows, 2 general rows.  R: rows per warp.
// Returns nullptr for a combination that is not instantiated.
MainKernel main_kernel_f16(int out_f32, int variant, int R);
MainKernel main_kernel_bf16(int out_f32, int variant, int R);
// Tiles kernel: aligned = 1 for the single-class fast path; (R, U) in
// {(1,8), (1,4), (2,4), (4,2)}.
// epi = 1 selects the copy built with the fused epilogue.
MainKernel tiles_kernel_f16(int out_f32, int aligned, int R, int U, int epi);
MainKernel tiles_kernel_bf16(int out_f32, int aligned, int R, int U, int epi);
// Bulk kernel (B staged through shared memory by bulk async copies): R = 1,
// unroll U in {4, 8} (32*U 16-byte blocks per ring buffer).
MainKernel bulk_kernel_f16(int out_f32, int aligned, int U, int epi);
MainKernel bulk_kernel_bf16(int out_f32, int aligned, int U, int epi);
ReduceKernel reduce_kernel_f16(int out_f32);
ReduceKernel reduce_kernel_bf16(int out_f32);

// Where a caller's buffer lives: every non-null pointer must start in
// device memory of `dev` (the current device) or in managed memory, which
// every device reaches.  Host memory (pinned, registered or pageable) and
// another device's memory give false.  One cudaPointerGetAttributes per
// pointer, no allocation, nothing launched.
inline bool on_device(int dev, std::initializer_list<const void *> ptrs) {
  for (const void *q : ptrs) {
    if (q == nullptr) continue;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (at.type == cudaMemoryTypeManaged) continue;
    if (at.type != cudaMemoryTypeDevice || at.device != dev) return false;
  }
  return true;
}

// Loads per lane issued back to back (per row) for R rows per warp.
inline int unroll_for_rows(int R) { return R == 1 ? 8 : (R == 2 ? 4 : 2); }

constexpr int kMaxThreads = 512;  // launch bound of the main kernel
constexpr int kFlagPrefetchB = 1;
constexpr int kFlagL2Shift = 1;  // 2 bits: tile rounds of bulk L2 prefetch ahead
constexpr int kFlagPrefetchA = 8;   // stage a before waiting on the predecessor
constexpr int kFlagEpilogue = 16;   // the fused epilogue is not the identity
constexpr int kFlagDeferStores = 32;  // tiles kernel with kFlagPrefetchA: keep row results, store after one wait
constexpr int kFlagL2First = 64;      // without kFlagPrefetchB: ask L2 for the first tile of B before the wait
constexpr int64_t kDeferMaxRows = 4096;  // most rows per CTA whose results are kept (16 KB of shared memory)
constexpr int kWaitPolls = 1 << 20;  // default bound on the polls of one mbarrier wait
constexpr uint32_t kDrainTimeoutBit = 0x80000000u;  // timeout counter: a drain of issued copies ran out

// Shared-memory layout of the bulk kernel, in bytes from the start of the
// dynamic allocation: staged a (as_elems * 2), slice partials (2 * W
// floats), then at a 128-byte boundary the W rings of `stages` buffers of
// 32 * U 16-byte blocks, then one 8-byte mbarrier per buffer.
GEMV_HD inline int64_t bulk_ring_offset(int64_t as_elems, int W) { return (as_elems * 2 + 8 * W + 127) / 128 * 128; }
GEMV_HD inline int64_t bulk_smem_bytes(int64_t as_elems, int W, int U, int stages) {
  return bulk_ring_offset(as_elems, W) + (int64_t)W * stages * (512 * U + 8);
}

}  // namespace gemvk

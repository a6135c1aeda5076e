// Native measurements that stand beside the GEMV benchmark, outside the
// library's ABI:
//
//  * host: the host cost of one cached gemv() call (validation, the
//    plan-cache lookup, one kernel launch) next to the cost of launching an
//    empty kernel on the same stream -- the floor any launch pays.  10^4
//    enqueues in bursts of 200 (so the launch queue never fills),
//    steady_clock around each burst, median over the bursts.
//  * read ceiling: a read-only streaming pass over two device buffers in
//    turn, with 32-byte non-coherent, no-L1-allocate loads (8 in flight per
//    thread; they measured 1-4 % faster than 16-byte ones) and nothing else
//    per CTA, timed back to back with CUDA events after a queue prefill --
//    as plain launches, and as programmatic dependent launches that never
//    wait (the buffers are never written, so consecutive passes may overlap
//    completely: the most a read-only stream of these bytes reaches on this
//    GPU).  Measured at 1 GiB per pass and at the bytes of one GEMV call's
//    B.
//
// Usage: gemv_bench_tool [gemv_b_bytes]   (default 234881024: 7168 x 16384 fp16)
// Prints one JSON line; exit status 0 on success.  Every kernel here ends by
// itself: the prefill spins for a fixed number of clock cycles.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "gemv.h"

namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeUnroll = 8;
constexpr uint32_t kProbeNever = 0x9e3779b9u;  // the sink is written only if a CTA's fold equals this

__global__ void empty_kernel() {}

// Keep the GPU busy for `cycles` SM clock cycles, so that the launches
// enqueued behind it are all queued before the timed region starts.
__global__ void spin_kernel(long long cycles) {
  const long long t0 = clock64();
  while (clock64() - t0 < cycles) {
  }
}

// 32 bytes at p (32-byte aligned), folded into one word.
__device__ __forceinline__ uint32_t ldg_stream32(const uint4 *p) {
  uint32_t r0, r1, r2, r3, r4, r5, r6, r7;
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3), "=r"(r4), "=r"(r5), "=r"(r6), "=r"(r7)
               : "l"(p));
  return r0 ^ r1 ^ r2 ^ r3 ^ r4 ^ r5 ^ r6 ^ r7;
}

// Grid-stride read of n32 32-byte units (unit j = 16-byte vectors 2j and
// 2j + 1), kProbeUnroll loads per thread in flight, folded into one word
// per thread; the word is stored (sink[blockIdx.x]) only if it equals
// kProbeNever, so the loads cannot be dropped and nothing else runs per
// CTA.  Under a programmatic dependent launch it lets its successor start at
// once and never waits for its predecessor.
__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4 *buf, int64_t n32, uint32_t *sink) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint32_t x = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kProbeUnroll - 1) * stride < n32; i += kProbeUnroll * stride) {
    uint32_t v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) v[u] = ldg_stream32(buf + 2 * (i + u * stride));
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) x ^= v[u];
  }
  for (; i < n32; i += stride) x ^= ldg_stream32(buf + 2 * i);
  if (x == kProbeNever) sink[blockIdx.x] = x;
}

template <class F>
double median_us_per_call(F &&fn, cudaStream_t s) {
  constexpr int kBursts = 50, kPerBurst = 200;
  std::vector<double> v;
  for (int b = 0; b < kBursts; ++b) {
    const auto t0 = std::chrono::steady_clock::now();
    for (int i = 0; i < kPerBurst; ++i) fn();
    const auto t1 = std::chrono::steady_clock::now();
    v.push_back(std::chrono::duration<double, std::micro>(t1 - t0).count() / kPerBurst);
    cudaStreamSynchronize(s);
  }
  std::sort(v.begin(), v.end());
  return v[v.size() / 2];
}

bool ok(cudaError_t e, const char *what) {
  if (e != cudaSuccess) {
    std::fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return false;
  }
  return true;
}

// Back-to-back read passes over bufs[0], bufs[1], ... in turn, `bytes` each
// (a multiple of 32); returns GB/s over `passes` timed passes (-1 on error).
double read_ceiling(uint4 *const bufs[2], int64_t bytes, int passes, bool pdl, int grid, uint32_t *sink,
                    cudaStream_t s, long long spin_cycles) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid);
  lc.blockDim = dim3(kProbeThreads);
  lc.stream = s;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  const int64_t n32 = bytes / 32;
  auto pass = [&](int i) { return cudaLaunchKernelEx(&lc, read_probe_kernel, (const uint4 *)bufs[i & 1], n32, sink); };
  for (int i = 0; i < 6; ++i)
    if (!ok(pass(i), "probe warm-up")) return -1;
  if (!ok(cudaStreamSynchronize(s), "probe warm-up sync")) return -1;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  spin_kernel<<<1, 1, 0, s>>>(spin_cycles);
  cudaEventRecord(e0, s);
  for (int i = 0; i < passes; ++i)
    if (!ok(pass(i), "probe pass")) return -1;
  cudaEventRecord(e1, s);
  if (!ok(cudaStreamSynchronize(s), "probe sync")) return -1;
  float ms = 0.f;
  cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return (double)bytes * passes / (ms * 1e-3) / 1e9;
}

}  // namespace

int main(int argc, char **argv) {
  const int64_t gemv_b_bytes = argc > 1 ? std::atoll(argv[1]) / 32 * 32 : 234881024;
  const int64_t n = 256, k = 512;  // the smallest workload shape
  void *B = nullptr, *a = nullptr, *c = nullptr;
  cudaStream_t s = nullptr;
  if (!ok(cudaMalloc(&B, n * k * 2), "cudaMalloc") || !ok(cudaMalloc(&a, k * 2), "cudaMalloc") ||
      !ok(cudaMalloc(&c, n * 2), "cudaMalloc") ||
      !ok(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking), "stream"))
    return 1;
  cudaMemset(B, 0, n * k * 2);
  cudaMemset(a, 0, k * 2);
  if (gemv(B, a, c, n, k, GEMV_F16, s) != GEMV_OK) return 2;  // plans and caches the launch
  cudaStreamSynchronize(s);
  int bad = 0;
  const double g = median_us_per_call([&] { bad |= gemv(B, a, c, n, k, GEMV_F16, s) != GEMV_OK; }, s);
  const double e = median_us_per_call([&] { empty_kernel<<<1, 32, 0, s>>>(); }, s);
  if (bad || !ok(cudaStreamSynchronize(s), "host-overhead sync")) return 3;

  // Read ceiling: two buffers of 1 GiB (and two of one GEMV call's B bytes).
  int dev = 0, sms = 0, per_sm = 0, clock_khz = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, dev);
  if (!ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, read_probe_kernel, kProbeThreads, 0), "occupancy"))
    return 4;
  const int grid = sms * (per_sm > 0 ? per_sm : 1);
  const int64_t big = 1LL << 30;
  uint4 *bufs[2] = {nullptr, nullptr};
  uint32_t *sink = nullptr;
  if (!ok(cudaMalloc(&bufs[0], big), "cudaMalloc") || !ok(cudaMalloc(&bufs[1], big), "cudaMalloc") ||
      !ok(cudaMalloc(&sink, 2 * grid * sizeof(uint32_t)), "cudaMalloc"))
    return 5;
  cudaMemset(bufs[0], 0x3c, big);
  cudaMemset(bufs[1], 0x5a, big);
  const long long spin = (long long)clock_khz * 2;  // ~2 ms at the rated clock
  const double r_big_plain = read_ceiling(bufs, big, 40, false, grid, sink, s, spin);
  const double r_big_pdl = read_ceiling(bufs, big, 40, true, grid, sink, s, spin);
  const int64_t small = std::min(gemv_b_bytes, big);
  const double r_small_plain = read_ceiling(bufs, small, 200, false, grid, sink, s, spin);
  const double r_small_pdl = read_ceiling(bufs, small, 200, true, grid, sink, s, spin);
  const bool fine = r_big_plain > 0 && r_big_pdl > 0 && r_small_plain > 0 && r_small_pdl > 0 &&
                    cudaGetLastError() == cudaSuccess;
  std::printf(
      "{\"gemv_us\": %.3f, \"empty_launch_us\": %.3f, \"calls\": 10000, \"n\": %lld, \"k\": %lld, "
      "\"read_gbs_1gib_plain\": %.1f, \"read_gbs_1gib_overlapped\": %.1f, \"read_bytes_small\": %lld, "
      "\"read_gbs_small_plain\": %.1f, \"read_gbs_small_overlapped\": %.1f, \"probe_grid\": %d}\n",
      g, e, (long long)n, (long long)k, r_big_plain, r_big_pdl, (long long)small, r_small_plain, r_small_pdl,
      grid);
  cudaFree(bufs[0]);
  cudaFree(bufs[1]);
  cudaFree(sink);
  cudaFree(B);
  cudaFree(a);
  cudaFree(c);
  cudaStreamDestroy(s);
  return fine ? 0 : 6;
}

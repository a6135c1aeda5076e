// Native measurements that stand beside the GEMV benchmark, outside the
// library's ABI:
//
//  * host: the host cost of one cached gemv() call (validation, the
//    plan-cache lookup, one kernel launch) next to the cost of launching an
//    empty kernel on the same stream -- the floor any launch pays.  10^4
//    enqueues in bursts of 200 (so the launch queue never fills),
//    steady_clock around each burst, median over the bursts.
//  * read ceiling: a read-only streaming pass over two device buffers in
//    turn, through the same 16-byte non-coherent, no-L1-allocate loads as
//    the GEMV kernels, timed back to back with CUDA events after a queue
//    prefill -- as plain launches, and as programmatic dependent launches
//    that never wait (the buffers are never written, so consecutive passes
//    may overlap completely: the most a read-only stream of these bytes
//    reaches on this GPU).  Measured at 1 GiB per pass and at the bytes of
//    one GEMV call's B.
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

__global__ void empty_kernel() {}

// Keep the GPU busy for `cycles` SM clock cycles, so that the launches
// enqueued behind it are all queued before the timed region starts.
__global__ void spin_kernel(long long cycles) {
  const long long t0 = clock64();
  while (clock64() - t0 < cycles) {
  }
}

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Grid-stride read of nvec 16-byte vectors, kProbeUnroll loads per thread
// in flight, folded into one XOR word per CTA (written to sink[blockIdx.x]
// so the loads cannot be dropped).  Under a programmatic dependent launch it
// lets its successor start at once and never waits for its predecessor.
__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4 *buf, int64_t nvec,
                                                                   uint32_t *sink) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint32_t x = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kProbeUnroll - 1) * stride < nvec; i += kProbeUnroll * stride) {
    uint4 v[kProbeUnroll];
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) v[u] = ldg_stream(buf + i + u * stride);
#pragma unroll
    for (int u = 0; u < kProbeUnroll; ++u) x ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < nvec; i += stride) {
    const uint4 v = ldg_stream(buf + i);
    x ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, m);
  __shared__ uint32_t part[kProbeThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t y = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) y ^= part[w];
    sink[blockIdx.x] = y;
  }
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
// (a multiple of 16); returns GB/s over `passes` timed passes (-1 on error).
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
  const int64_t nvec = bytes / 16;
  auto pass = [&](int i) {
    return cudaLaunchKernelEx(&lc, read_probe_kernel, (const uint4 *)bufs[i & 1], nvec, sink + (i & 1) * grid);
  };
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
  const int64_t gemv_b_bytes = argc > 1 ? std::atoll(argv[1]) / 16 * 16 : 234881024;
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

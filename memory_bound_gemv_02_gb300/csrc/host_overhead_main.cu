// Native measurement of the host cost of one cached gemv() call (the launch
// path only: validation, plan-cache lookup, one kernel launch), next to the
// cost of launching an empty kernel on the same stream -- the floor any
// launch pays.  10^4 enqueues in bursts of 200 (so the launch queue never
// fills), steady_clock around each burst, median over the bursts.  Prints
// one JSON line.  Exit status 0 on success.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <vector>

#include "gemv.h"

namespace {

__global__ void empty_kernel() {}

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

}  // namespace

int main() {
  const int64_t n = 256, k = 512;  // the smallest workload shape
  void *B = nullptr, *a = nullptr, *c = nullptr;
  cudaStream_t s = nullptr;
  if (cudaMalloc(&B, n * k * 2) != cudaSuccess || cudaMalloc(&a, k * 2) != cudaSuccess ||
      cudaMalloc(&c, n * 2) != cudaSuccess || cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    std::fprintf(stderr, "CUDA setup failed\n");
    return 1;
  }
  cudaMemset(B, 0, n * k * 2);
  cudaMemset(a, 0, k * 2);
  if (gemv(B, a, c, n, k, GEMV_F16, s) != GEMV_OK) return 2;  // plans and caches the launch
  cudaStreamSynchronize(s);
  int bad = 0;
  const double g = median_us_per_call([&] { bad |= gemv(B, a, c, n, k, GEMV_F16, s) != GEMV_OK; }, s);
  const double e = median_us_per_call([&] { empty_kernel<<<1, 32, 0, s>>>(); }, s);
  const bool ok = !bad && cudaStreamSynchronize(s) == cudaSuccess && cudaGetLastError() == cudaSuccess;
  std::printf("{\"gemv_us\": %.3f, \"empty_launch_us\": %.3f, \"calls\": 10000, \"n\": %lld, \"k\": %lld}\n", g, e,
              (long long)n, (long long)k);
  cudaFree(B);
  cudaFree(a);
  cudaFree(c);
  cudaStreamDestroy(s);
  return ok ? 0 : 3;
}

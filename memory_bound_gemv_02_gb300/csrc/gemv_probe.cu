// Read-only bandwidth probe: streams a buffer through the same 16-byte
// non-coherent, no-L1-allocate load path as the GEMV kernels and folds it
// into one XOR checksum per CTA.  It calibrates the achievable HBM read
// rate; it is not part of the product path.
#include "gemv_kernels.cuh"

namespace gemvk {

__global__ void __launch_bounds__(512) gemv_probe_kernel(const uint4 *buf, int64_t nvec, uint32_t *sink) {
  constexpr int U = 8;
  uint32_t x = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (U - 1) * stride < nvec; i += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ldg_stream(buf + i + u * stride);
#pragma unroll
    for (int u = 0; u < U; ++u) x ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < nvec; i += stride) {
    const uint4 v = ldg_stream(buf + i);
    x ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, m);
  __shared__ uint32_t part[kMaxThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t y = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) y ^= part[w];
    sink[blockIdx.x] = y;
  }
}

ProbeKernel probe_kernel() { return gemv_probe_kernel; }

}  // namespace gemvk

// Reductions of the blend's quality diagnostics ("数学推导" §形式化: the attention deviation
// ||Attention(Q, K_fused, V_fused) - Attention(Q, K_new, V_new)||; §注意力稀疏性的量化分析:
// Sparsity(A, eps) = |{(i, j): A_ij < eps}| / n^2). The per-row counts come from the counting
// instance of the attention kernel; these kernels only add up.
#include "common.cuh"
#include "kernels.h"

namespace cb {

namespace {

constexpr int kRedThreads = 256;

__global__ void __launch_bounds__(kRedThreads) sum_counts_kernel(const int32_t* __restrict__ counts, int64_t n,
                                                                 unsigned long long* total) {
  pdl_launch_dependents();
  pdl_wait();
  unsigned long long acc = 0;
  for (int64_t i = blockIdx.x * (int64_t)kRedThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kRedThreads)
    acc += (unsigned long long)counts[i];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (threadIdx.x % 32 == 0 && acc != 0) atomicAdd(total, acc);
}

__global__ void __launch_bounds__(kRedThreads) output_deviation_kernel(const uint8_t* __restrict__ a,
                                                                       const uint8_t* __restrict__ b, int64_t n8,
                                                                       double* sums) {
  pdl_launch_dependents();
  pdl_wait();
  double d2 = 0.0, r2 = 0.0;
  for (int64_t i = blockIdx.x * (int64_t)kRedThreads + threadIdx.x; i < n8; i += (int64_t)gridDim.x * kRedThreads) {
    float x[8], y[8];
    unpack8(ld_stream(a + i * 16), x);
    unpack8(ld_stream(b + i * 16), y);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const double d = (double)x[e] - (double)y[e];
      d2 = fma(d, d, d2);
      r2 = fma((double)y[e], (double)y[e], r2);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    d2 += __shfl_xor_sync(0xffffffffu, d2, off);
    r2 += __shfl_xor_sync(0xffffffffu, r2, off);
  }
  __shared__ double s[2][kRedThreads / 32];
  if (threadIdx.x % 32 == 0) {
    s[0][threadIdx.x / 32] = d2;
    s[1][threadIdx.x / 32] = r2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double t0 = 0.0, t1 = 0.0;
    for (int w = 0; w < kRedThreads / 32; ++w) {
      t0 += s[0][w];
      t1 += s[1][w];
    }
    atomicAdd(&sums[0], t0);
    atomicAdd(&sums[1], t1);
  }
}

int grid_for(int64_t items) {
  int64_t b = (items + kRedThreads - 1) / kRedThreads;
  return (int)(b < 1 ? 1 : (b > 152 * 4 ? 152 * 4 : b));
}

}  // namespace

cudaError_t launch_sum_counts(const int32_t* counts, int64_t n, unsigned long long* total, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(total, 0, sizeof(unsigned long long), s);
  if (e != cudaSuccess || n <= 0) return e;
  return launch_pdl(sum_counts_kernel, grid_for(n), kRedThreads, 0, s, counts, n, total);
}

cudaError_t launch_output_deviation(const void* a, const void* b, int64_t n, double* sums, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(sums, 0, 2 * sizeof(double), s);
  if (e != cudaSuccess || n <= 0) return e;
  return launch_pdl(output_deviation_kernel, grid_for(n / 8), kRedThreads, 0, s, (const uint8_t*)a,
                    (const uint8_t*)b, n / 8, sums);
}

}  // namespace cb

// Microbenchmark of the arithmetic units the softmax runs on, the secondary
// roofs of the attention kernels next to the tensor pipe: the MUFU exp2
// (ex2.approx, one per score in the forward and in the backward's P), and
// the FP32 pipe (FFMA, and the packed two-lane FFMA2 the forward's softmax
// uses). Not part of the method; it measures the hardware it runs on.
//
// Each pipe gets one kernel: 2 blocks of 1024 threads per SM (one full wave,
// every warp slot used), each thread running 8 independent dependency chains
// of the instruction for `iters` rounds between two clock64 reads, each after
// a block barrier. Thread 0 of every block records the block's cycle count;
// the largest over the grid bounds the time the SM's 2 x 1024 x 8 x iters
// operations took.

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRateThreads = 1024;
constexpr int kRateChains = 8;

// pipe: 0 = ex2.approx.ftz.f32, 1 = fma.rn.f32, 2 = fma.rn.f32x2 (two lanes)
template <int PIPE>
__global__ void __launch_bounds__(kRateThreads, 2)
    unit_rate_kernel(unsigned long long* cycles, int iters, float seed) {
  float x[kRateChains], y[kRateChains];
#pragma unroll
  for (int c = 0; c < kRateChains; ++c) {
    x[c] = seed * static_cast<float>((threadIdx.x + c) & 7) * 0.125f;
    y[c] = 1.f - x[c];
  }
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kRateChains; ++c) {
      if constexpr (PIPE == 0) {
        // the form the attention kernels use; its timing does not depend on
        // the values, which run off to +inf
        asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(x[c]));
      } else if constexpr (PIPE == 1) {
        asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x[c]) : "f"(0.999f), "f"(1e-4f));
      } else {
        const float2 r = ffma2(make_float2(x[c], y[c]), make_float2(0.999f, 0.999f),
                               make_float2(1e-4f, 1e-4f));
        x[c] = r.x;
        y[c] = r.y;
      }
    }
  }
  // every warp of the block has finished before the end time is read, so
  // that thread 0's span covers the block's work
  __syncthreads();
  const unsigned long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < kRateChains; ++c) acc += x[c] + y[c];
  if (threadIdx.x == 0) {
    atomicMax(cycles, t1 - t0);
    if (acc == 12345.f) atomicAdd(cycles + 1, 1ull);  // keeps the chains live
  }
}

}  // namespace

cudaError_t launch_unit_rates(unsigned long long* cycles, int iters, int num_sms,
                              cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(cycles, 0, 6 * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  const dim3 grid(2 * num_sms);
  unit_rate_kernel<0><<<grid, kRateThreads, 0, stream>>>(cycles, iters, 0.5f);
  unit_rate_kernel<1><<<grid, kRateThreads, 0, stream>>>(cycles + 2, iters, 0.5f);
  unit_rate_kernel<2><<<grid, kRateThreads, 0, stream>>>(cycles + 4, iters, 0.5f);
  return cudaGetLastError();
}

}  // namespace fa

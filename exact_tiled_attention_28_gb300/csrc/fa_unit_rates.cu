// Microbenchmark of the arithmetic units the softmax runs on, the secondary
// roofs of the attention kernels next to the tensor pipe: the MUFU exp2
// (ex2.approx, one per score in the forward and in the backward's P), and
// the FP32 pipe (FFMA, and the packed two-lane FFMA2 the forward's softmax
// uses). Not part of the method; it measures the hardware it runs on.
//
// Each pipe gets one kernel: 2 blocks of 1024 threads per SM (one full wave,
// every warp slot used), each thread running 8 independent dependency chains
// of the instruction for `iters` rounds between two clock64 reads, each after
// a block barrier. Thread 0 of every block folds its start and end into its
// SM's earliest start and latest end (the SM's clock is one counter for both
// blocks, which need not start together); the longest such span over the SMs
// bounds the time an SM's 2 x 1024 x 8 x iters operations took. Timing each
// block alone missed the skew between the two blocks' starts: FFMA then read
// up to 131 per clock per SM, above the 128 lanes an SM has.

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRateThreads = 1024;
constexpr int kRateChains = 8;
constexpr int kRateMaxSms = 256;  // %smid values past this are not recorded

// [pipe][earliest start, latest end][SM]
__device__ unsigned long long g_rate_span[3][2][kRateMaxSms];

__global__ void rate_span_init_kernel() {
  const int i = threadIdx.x;
  if (i < kRateMaxSms) {
    for (int p = 0; p < 3; ++p) {
      g_rate_span[p][0][i] = ~0ull;
      g_rate_span[p][1][i] = 0ull;
    }
  }
}

// cycles[2 p] = the longest SM span of pipe p
__global__ void rate_span_final_kernel(unsigned long long* cycles) {
  __shared__ unsigned long long best[3];
  if (threadIdx.x < 3) best[threadIdx.x] = 0ull;
  __syncthreads();
  const int i = threadIdx.x;
  if (i < kRateMaxSms) {
    for (int p = 0; p < 3; ++p) {
      const unsigned long long t0 = g_rate_span[p][0][i], t1 = g_rate_span[p][1][i];
      if (t0 != ~0ull && t1 > t0) atomicMax(&best[p], t1 - t0);
    }
  }
  __syncthreads();
  if (threadIdx.x < 3) cycles[2 * threadIdx.x] = best[threadIdx.x];
}

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
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    if (smid < kRateMaxSms) {
      atomicMin(&g_rate_span[PIPE][0][smid], t0);
      atomicMax(&g_rate_span[PIPE][1][smid], t1);
    }
    if (acc == 12345.f) atomicAdd(cycles + 1, 1ull);  // keeps the chains live
  }
}

}  // namespace

cudaError_t launch_unit_rates(unsigned long long* cycles, int iters, int num_sms,
                              cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(cycles, 0, 6 * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  rate_span_init_kernel<<<1, kRateMaxSms, 0, stream>>>();
  const dim3 grid(2 * num_sms);
  unit_rate_kernel<0><<<grid, kRateThreads, 0, stream>>>(cycles, iters, 0.5f);
  unit_rate_kernel<1><<<grid, kRateThreads, 0, stream>>>(cycles + 2, iters, 0.5f);
  unit_rate_kernel<2><<<grid, kRateThreads, 0, stream>>>(cycles + 4, iters, 0.5f);
  rate_span_final_kernel<<<1, kRateMaxSms, 0, stream>>>(cycles);
  return cudaGetLastError();
}

}  // namespace fa

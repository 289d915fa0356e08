// fa_bwd_noalloc: the backward for callers that cannot allocate device memory.
//
// Who needs it: a caller whose device memory is all handed to its own pool
// (so there is nothing left for it to cudaMalloc a workspace from), or one
// that must not call cudaMalloc once it is running, because cudaMalloc can
// synchronise the whole device and takes an unbounded time. fa_bwd needs a
// caller-provided workspace; this variant uses a fixed array that lives in the
// library's own device image instead, so the caller passes only its inputs
// and outputs and nothing is allocated by anyone at call time.
//
// The array is file-scope device memory of FA_NOALLOC_SCRATCH_BYTES (32 MiB).
// Every GPU that loads this library holds it until the process exits. All
// calls share it and it keeps the last call's contents; the backward's first
// stage rewrites every part of it that later stages read (it zeroes the dQ
// accumulator and writes the D and log-sum-exp rows), so nothing has to be
// cleared beforehand. Two calls that run on the GPU at the same time (other
// streams, other host threads) race on the array and give wrong results.

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "kernels.h"

namespace fa {

// device info of the current device (defined in fa_api.cu)
cudaError_t current_device_setup(int* num_sms, int** status);

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// The device address of the scratch array on the current device. In host
// code g_noalloc_scratch names a host-side stand-in, not device memory, so the
// address has to come from cudaGetSymbolAddress, once per device, with that
// device current. The first call on each device does this.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dO, void* dq, void* dk,
                                    void* dv, int B, int H, int N, int d, int causal,
                                    float scale, void* stream) {
  // the same argument rules as fa_bwd, checked before anything is enqueued
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    return FA_ERR_UNSUPPORTED;  // head dimension, or B*H too large
  }
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, o, static_cast<const void*>(lse), dO,
                        static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if (p == nullptr || !fa::aligned16(p)) return FA_ERR_INVALID_ARG;
  // sizes whose workspace does not fit in the fixed array are refused
  if (need > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES)) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (fa::scratch_address(&scratch) != cudaSuccess) return FA_ERR_CUDA;
  int num_sms = 0;
  int* status = nullptr;
  if (fa::current_device_setup(&num_sms, &status) != cudaSuccess) return FA_ERR_CUDA;
  fa::Problem p{B, H, N, d, causal ? 1 : 0, scale, num_sms, status, {}};
  for (int t = 0; t < fa::kNumTensors; ++t) p.st[t] = fa::contiguous_strides(H, N, d);
  const cudaError_t e = fa::launch_bwd(p, q, k, v, o, lse, dO, dq, dk, dv, scratch,
                                       fa::kStagesAll, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

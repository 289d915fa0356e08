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
// Every GPU on which any entry point of this library has been called holds it
// until the process exits: CUDA loads a library's device code lazily, per
// device, and the library forces that load (and so the reservation of the
// array) at its first call on each device, whichever entry point it is. All
// calls share it and it keeps the last call's contents; the backward's first
// stage rewrites every part of it that later stages read (it zeroes the dQ
// accumulator and writes the D and log-sum-exp rows), so nothing has to be
// cleared beforehand. Two calls that run on the GPU at the same time (other
// streams, other host threads) race on the array and give wrong results.

#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "kernels.h"

namespace fa {

// device facts of the current device (fa_api.cu): the SM count, the status
// word and this file's scratch array, all as device addresses
cudaError_t current_device_setup(int* num_sms, int** status, void** scratch);

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// The device address of the scratch array on the current device. In host code
// g_noalloc_scratch names a host-side stand-in, not device memory, so the
// address has to come from cudaGetSymbolAddress with the device current. The
// library's per-device set-up (fa_api.cu) calls this at the first call of any
// entry point on a device, and again in a new context after cudaDeviceReset.
cudaError_t noalloc_scratch_lookup(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  *out = p;
  return cudaSuccess;
}

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
  int num_sms = 0;
  int* status = nullptr;
  void* scratch = nullptr;
  if (fa::current_device_setup(&num_sms, &status, &scratch) != cudaSuccess) return FA_ERR_CUDA;
  fa::Problem p{B, H, N, d, causal ? 1 : 0, scale, num_sms, status, {}};
  for (int t = 0; t < fa::kNumTensors; ++t) p.st[t] = fa::contiguous_strides(H, N, d);
  const cudaError_t e = fa::launch_bwd(p, q, k, v, o, lse, dO, dq, dk, dv, scratch,
                                       fa::kStagesAll, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

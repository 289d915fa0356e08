// The C ABI of libfa.so (declared in include/fa.h): argument checks, TMA
// descriptor encoding, the device status word, and the launches.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/fa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fa {

// The status word of every kernel in this library; a bounded wait that runs
// out records DEV_TIMEOUT here.
__device__ int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device set-up, done once with that device current.
cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return e;
    di.status = static_cast<int*>(p);
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess) return e;
      if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    di.ready = true;
  }
  *out = di;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_sizes(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H >= (int64_t(1) << 31)) return FA_ERR_UNSUPPORTED;
  if (d != 32 && d != 64 && d != 96 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || scale < 0.f) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Strides (in elements) of a [B, H, N, d] tensor whose rows hold d
// contiguous values: positive multiples of 8 (16 bytes, for TMA and 16-byte
// stores), rows at least d apart, below 2^36 elements.
fa_status check_strides(const long long* st, int n) {
  if (st == nullptr) return FA_ERR_INVALID_ARG;
  for (int i = 0; i < 3 * n; ++i)
    if (st[i] <= 0 || (st[i] & 7) != 0 || st[i] >= (1ll << 36)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// One thread waits on a barrier that nothing arrives on, with the given
// limit; the bounded wait gives up, records DEV_TIMEOUT and the kernel returns.
__global__ void wait_timeout_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  mbar_init(smem_u32(&bar), 1);
  abort_flag = 0;
  fence_barrier_init();
  mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

// Evaluates the forward kernel's FMA-pipe exp2 on n inputs.
__global__ void exp2_selftest_kernel(const float* x, float* y, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i + 1 < n) {
    const float2 r = exp2_poly2(make_float2(x[i], x[i + 1]));
    y[i] = r.x;
    y[i + 1] = r.y;
  } else if (i < n) {
    y[i] = exp2_poly2(make_float2(x[i], x[i])).x;
  }
}

}  // namespace

// Device facts for launchers outside this file (the no-alloc entry point).
cudaError_t current_device_setup(int* num_sms, int** status) {
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  *num_sms = di.num_sms;
  *status = di.status;
  return cudaSuccess;
}

bool make_tile_map(CUtensorMap* map, const void* base, int B, int H, int N, int d,
                   const Strides& s) {
  if (!g_encode) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.row) * 2,
                                 static_cast<cuuint64_t>(s.head) * 2,
                                 static_cast<cuuint64_t>(s.batch) * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kTile), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa

extern "C" {

int fa_abi_version(void) { return 1; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null or misaligned pointer, size < 1 or bad scale";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dimension must be 32, 64, 96 or 128";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side bounded wait expired";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: backward workspace null or too small";
    default: return "unknown fa_status";
  }
}

namespace {

// strides: 3 per tensor (batch, head, row) in TensorId order, or null for
// contiguous [B, H, N, d] tensors
fa_status fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, const long long* strides, int causal, float scale,
                     void* stream) {
  fa_status s = fa::check_sizes(B, H, N, d, scale);
  if (s != FA_OK) return s;
  s = fa::check_ptrs({q, k, v, o, lse});
  if (s != FA_OK) return s;
  if (strides != nullptr) {
    s = fa::check_strides(strides, 4);
    if (s != FA_OK) return s;
  }
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return FA_ERR_CUDA;
  fa::Problem p{B, H, N, d, causal ? 1 : 0, scale, di.num_sms, di.status, {}};
  for (int t = 0; t < fa::kNumTensors; ++t)
    p.st[t] = (strides != nullptr && t < 4)
                  ? fa::Strides{strides[3 * t], strides[3 * t + 1], strides[3 * t + 2]}
                  : fa::contiguous_strides(H, N, d);
  const cudaError_t e = fa::launch_fwd(p, q, k, v, o, lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, int causal, float scale, void* stream) {
  return fwd_common(q, k, v, o, lse, B, H, N, d, nullptr, causal, scale, stream);
}

fa_status fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, const long long* strides, int causal, float scale,
                         void* stream) {
  if (strides == nullptr) return FA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, B, H, N, d, strides, causal, scale, stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (fa::check_sizes(B, H, N, d, 1.f) != FA_OK) return 0;
  return fa::bwd_workspace_bytes(B, H, N, d);
}

namespace {

fa_status bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                     int causal, float scale, void* workspace, size_t workspace_bytes, int stages,
                     std::initializer_list<const void*> used, void* stream,
                     const long long* strides = nullptr) {
  fa_status s = fa::check_sizes(B, H, N, d, scale);
  if (s != FA_OK) return s;
  s = fa::check_ptrs(used);
  if (s != FA_OK) return s;
  if (strides != nullptr) {
    s = fa::check_strides(strides, fa::kNumTensors);
    if (s != FA_OK) return s;
  }
  if (workspace == nullptr || !fa::aligned16(workspace) ||
      workspace_bytes < fa::bwd_workspace_bytes(B, H, N, d))
    return FA_ERR_WORKSPACE;
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return FA_ERR_CUDA;
  fa::Problem p{B, H, N, d, causal ? 1 : 0, scale, di.num_sms, di.status, {}};
  for (int t = 0; t < fa::kNumTensors; ++t)
    p.st[t] = strides != nullptr ? fa::Strides{strides[3 * t], strides[3 * t + 1], strides[3 * t + 2]}
                                 : fa::contiguous_strides(H, N, d);
  const cudaError_t e = fa::launch_bwd(p, q, k, v, o, lse, dO, dq, dk, dv, workspace, stages,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, workspace,
                    workspace_bytes, fa::kStagesAll, {q, k, v, o, lse, dO, dq, dk, dv}, stream);
}

fa_status fa_bwd_strided(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, const long long* strides, int causal, float scale,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (strides == nullptr) return FA_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, workspace,
                    workspace_bytes, fa::kStagesAll, {q, k, v, o, lse, dO, dq, dk, dv}, stream,
                    strides);
}

fa_status fa_bwd_preprocess(const void* o, const float* lse, const void* dO, int B, int H, int N,
                            int d, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(nullptr, nullptr, nullptr, o, lse, dO, nullptr, nullptr, nullptr, B, H, N, d,
                    0, 1.f, workspace, workspace_bytes, fa::kStagePre, {o, lse, dO}, stream);
}

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                      void* dv, int B, int H, int N, int d, int causal, float scale,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(q, k, v, nullptr, nullptr, dO, nullptr, dk, dv, B, H, N, d, causal, scale,
                    workspace, workspace_bytes, fa::kStageDkdv, {q, k, v, dO, dk, dv}, stream);
}

fa_status fa_bwd_dq_finalize(void* dq, int B, int H, int N, int d, float scale, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return bwd_common(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr, nullptr, B,
                    H, N, d, 0, scale, workspace, workspace_bytes, fa::kStageDq, {dq}, stream);
}

fa_status fa_selftest_wait_timeout(int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 2000) return FA_ERR_INVALID_ARG;
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return FA_ERR_CUDA;
  fa::wait_timeout_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      di.status, static_cast<uint64_t>(limit_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_selftest_exp2(const float* x, float* y, int n, void* stream) {
  if (x == nullptr || y == nullptr || n < 1) return FA_ERR_INVALID_ARG;
  const int threads = 256, blocks = (n / 2 + threads) / threads;
  fa::exp2_selftest_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_last_device_status(void* stream) {
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return FA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, fa::g_device_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (h != fa::DEV_OK) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_device_status, &zero, sizeof(int)) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

}  // extern "C"

// The C ABI of libfa.so (declared in include/fa.h): argument checks, TMA
// descriptor encoding, the device status word, and the launches.

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstddef>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/fa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fa {

// The status word of every kernel in this library, with the bounded-wait
// limit beside it (ptx.cuh, DeviceWord); a bounded wait that runs out records
// DEV_TIMEOUT in the status member.
__device__ DeviceWord g_device_word = {DEV_OK, 0, kWaitLimitNs};

// Device address of the no-alloc backward's fixed scratch array
// (fa_noalloc.cu), looked up with the device current.
cudaError_t noalloc_scratch_lookup(void** out);

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  unsigned long long ctx_id = 0;  // the CUDA context the addresses below belong to
  int num_sms = 0;
  int* status = nullptr;
  void* scratch = nullptr;  // fa_bwd_noalloc's array
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

cudaError_t driver_entry(const char* name, unsigned version, void** fn) {
  cudaDriverEntryPointQueryResult q;
  const cudaError_t e = cudaGetDriverEntryPointByVersion(name, fn, version, cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || *fn == nullptr) return cudaErrorSymbolNotFound;
  return cudaSuccess;
}

// Unique id of the context current on this thread, 0 if none is current yet.
// Ids are never reused within a process, so a context made after
// cudaDeviceReset has a new one.
unsigned long long current_ctx_id() {
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Per-device set-up, done with that device current: the SM count, the device
// addresses of the status word and of the no-alloc scratch array, and the
// driver entry points. The addresses belong to the device's context, so the
// set-up is redone when the current context is not the one they were taken in
// (after cudaDeviceReset). Looking up the scratch array here, at the first
// call of any entry point on a device, is what loads the module that holds
// it: CUDA loads modules lazily by default, and the array's device memory is
// reserved at that load.
cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    if ((e = driver_entry("cuTensorMapEncodeTiled", 12000, &fn)) != cudaSuccess) return e;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    if ((e = driver_entry("cuCtxGetCurrent", 4000, &fn)) != cudaSuccess) return e;
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    if ((e = driver_entry("cuCtxGetId", 12000, &fn)) != cudaSuccess) return e;
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  }
  DeviceInfo& di = g_dev[dev];
  const unsigned long long ctx = current_ctx_id();
  if (!di.ready || ctx == 0 || ctx != di.ctx_id) {
    di.ready = false;
    e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_word);  // makes the device's context current
    if (e != cudaSuccess) return e;
    di.status = &static_cast<DeviceWord*>(p)->status;
    e = noalloc_scratch_lookup(&di.scratch);
    if (e != cudaSuccess) return e;
    di.ctx_id = current_ctx_id();
    di.ready = di.ctx_id != 0;
  }
  *out = di;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// allow256: the forward and backward of dense (or strided) equal-length
// batches also take d = 256; nothing else does. Their work items (query
// tiles in the forward, 64-key blocks in the backward) are counted in int.
fa_status check_sizes(int B, int H, int N, int d, float scale, bool allow256 = false) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H >= (int64_t(1) << 31)) return FA_ERR_UNSUPPORTED;
  if (d != 32 && d != 64 && d != 96 && d != 128 && !(allow256 && d == 256))
    return FA_ERR_UNSUPPORTED;
  if (allow256 && d == 256 &&
      static_cast<int64_t>(B) * H * ((static_cast<int64_t>(N) + 63) / 64) >= (int64_t(1) << 31))
    return FA_ERR_UNSUPPORTED;
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

// Checks a packed batch's sequence offsets (see launch_varlen_check).
__global__ void varlen_check_kernel(const int* cu_q, const int* cu_k, int B, int rows_q,
                                    int rows_k, int max_q, int max_k, int* status) {
  bool bad = false;
  for (int b = threadIdx.x; b <= B; b += blockDim.x) {
    const long long q = cu_q[b], k = cu_k[b];
    if (b == 0 && (q != 0 || k != 0)) bad = true;
    if (b == B && (q != rows_q || k != rows_k)) bad = true;
    if (b < B) {
      const long long nq = cu_q[b + 1] - q, nk = cu_k[b + 1] - k;
      if (nq < 0 || nk < 0 || nq > max_q || nk > max_k) bad = true;
    }
  }
  if (bad) atomicCAS(status, DEV_OK, DEV_BADARG);
}

// Checks per-sequence key counts (see launch_klens_check).
__global__ void klens_check_kernel(const int* lens, int B, int Nk, int* status) {
  bool bad = false;
  for (int b = threadIdx.x; b < B; b += blockDim.x) bad |= lens[b] < 0 || lens[b] > Nk;
  if (bad) atomicCAS(status, DEV_OK, DEV_BADARG);
}

// Debug build: one failed index check (on an index computed at run time from
// the lane number, so that the compiler cannot drop it); no memory is
// accessed.
__global__ void index_check_selftest_kernel(int* status) {
  const int idx = static_cast<int>(threadIdx.x) + 32;  // one past a 32-element range
  fa_dcheck(idx < 32, status);
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
cudaError_t current_device_setup(int* num_sms, int** status, void** scratch) {
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  *num_sms = di.num_sms;
  *status = di.status;
  *scratch = di.scratch;
  return cudaSuccess;
}

cudaError_t launch_klens_check(const int* lens, int B, int Nk, int* status, cudaStream_t stream) {
  klens_check_kernel<<<1, 256, 0, stream>>>(lens, B, Nk, status);
  return cudaGetLastError();
}

cudaError_t launch_varlen_check(const Problem& p, cudaStream_t stream) {
  varlen_check_kernel<<<1, 256, 0, stream>>>(p.cu_q, p.cu_k, p.B, p.rows_q, p.rows_k, p.max_q,
                                             p.max_k, p.status);
  return cudaGetLastError();
}

bool make_tile_map(CUtensorMap* map, const void* base, int B, int H, int N, int d,
                   const Strides& s, int box_rows, int box_blocks) {
  if (!g_encode) return false;
  if (box_blocks > 1) {
    if (d % 64 != 0 || box_blocks > d / 64) return false;
    const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(d / 64),
                                static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[4] = {static_cast<cuuint64_t>(s.row) * 2, 128,
                                   static_cast<cuuint64_t>(s.head) * 2,
                                   static_cast<cuuint64_t>(s.batch) * 2};
    const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(box_rows),
                               static_cast<cuuint32_t>(box_blocks), 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.row) * 2,
                                 static_cast<cuuint64_t>(s.head) * 2,
                                 static_cast<cuuint64_t>(s.batch) * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa

extern "C" {

int fa_abi_version(void) { return 2; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null or misaligned pointer, size < 1 or bad scale";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dimension or size not supported by this call";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side bounded wait expired";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: backward workspace null or too small";
    case FA_ERR_DEVICE_CHECK: return "FA_ERR_DEVICE_CHECK: a device-side index check failed (debug build)";
    default: return "unknown fa_status";
  }
}

namespace {

// strides: 3 per tensor (batch, head, row) in TensorId order, or null for
// contiguous [B, H, N, d] tensors
fa_status fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, const long long* strides, int causal, float scale,
                     void* stream) {
  fa_status s = fa::check_sizes(B, H, N, d, scale, /*allow256=*/true);
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
  if (fa::check_sizes(B, H, N, d, 1.f, /*allow256=*/true) != FA_OK) return 0;
  return fa::bwd_workspace_bytes(B, H, N, d);
}

namespace {

// The dQ path fa_bwd takes for a shape (FA_DQ_AUTO): the atomic one, which
// measured faster on GB300 in every case timed (see fa_bwd_with_dq_path).
bool auto_dq_separate(int /*B*/, int /*H*/, int /*N*/, int /*d*/, int /*causal*/) { return false; }

fa_status bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                     int causal, float scale, void* workspace, size_t workspace_bytes, int stages,
                     std::initializer_list<const void*> used, void* stream,
                     const long long* strides = nullptr, int dq_path = FA_DQ_AUTO) {
  fa_status s = fa::check_sizes(B, H, N, d, scale, /*allow256=*/true);
  if (s != FA_OK) return s;
  if (dq_path != FA_DQ_AUTO && dq_path != FA_DQ_ATOMIC && dq_path != FA_DQ_SEPARATE)
    return FA_ERR_INVALID_ARG;
  if (dq_path == FA_DQ_SEPARATE && !fa::bwd_dq_separate_supported(d)) return FA_ERR_UNSUPPORTED;
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
  p.dq_separate = dq_path == FA_DQ_SEPARATE ||
                  (dq_path == FA_DQ_AUTO && fa::bwd_dq_separate_supported(d) &&
                   auto_dq_separate(B, H, N, d, causal));
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

fa_status fa_bwd_with_dq_path(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dO, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal, float scale, int dq_path,
                              void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, workspace,
                    workspace_bytes, fa::kStagesAll, {q, k, v, o, lse, dO, dq, dk, dv}, stream,
                    nullptr, dq_path);
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

namespace {

// Work items of the var kernels must fit an int: sequences x heads x the
// longest sequence's tiles.
bool var_items_fit(int B, int H, int max_q, int max_k) {
  const int64_t bh = static_cast<int64_t>(B) * H;
  return bh * ((max_q + 255) / 256) < (int64_t(1) << 31) &&
         bh * ((max_k + 127) / 128) < (int64_t(1) << 31);
}

// Problem for B dense sequences of Nq query and Nk key rows; strides: 3 per
// tensor (batch, head, row) in TensorId order for n tensors, or null.
fa_status nqnk_problem(fa::Problem* p, int B, int H, int Nq, int Nk, int d,
                       const long long* strides, int n, int causal, float scale) {
  fa_status s = fa::check_sizes(B, H, Nq, d, scale);
  if (s != FA_OK) return s;
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  if (!var_items_fit(B, H, Nq, Nk)) return FA_ERR_UNSUPPORTED;
  if (strides != nullptr) {
    s = fa::check_strides(strides, n);
    if (s != FA_OK) return s;
  }
  *p = fa::Problem{B, H, Nq, d, causal ? 1 : 0, scale, 0, nullptr, {}};
  for (int t = 0; t < fa::kNumTensors; ++t) {
    const bool kv = t == fa::kK || t == fa::kV || t == fa::kdK || t == fa::kdV;
    p->st[t] = (strides != nullptr && t < n)
                   ? fa::Strides{strides[3 * t], strides[3 * t + 1], strides[3 * t + 2]}
                   : fa::contiguous_strides(H, kv ? Nk : Nq, d);
  }
  p->var = 1;
  p->Nk = Nk;
  p->rows_q = p->max_q = Nq;
  p->rows_k = p->max_k = Nk;
  return FA_OK;
}

// Problem for a packed batch; strides: 2 per tensor (head, row) for n
// tensors, or null for [T, H, d] tensors.
fa_status varlen_problem(fa::Problem* p, const int* cu_q, const int* cu_k, int B, int H,
                         int total_q, int total_k, int max_q, int max_k, int d,
                         const long long* strides, int n, int causal, float scale) {
  fa_status s = fa::check_sizes(B, H, total_q, d, scale);
  if (s != FA_OK) return s;
  if (total_k < 1 || max_q < 1 || max_k < 1 || cu_q == nullptr || cu_k == nullptr ||
      (reinterpret_cast<uintptr_t>(cu_q) & 3u) != 0 || (reinterpret_cast<uintptr_t>(cu_k) & 3u) != 0)
    return FA_ERR_INVALID_ARG;
  if (!var_items_fit(B, H, max_q, max_k)) return FA_ERR_UNSUPPORTED;
  long long st[3 * fa::kNumTensors];
  for (int t = 0; t < fa::kNumTensors; ++t) {
    const long long head = strides != nullptr && t < n ? strides[2 * t] : d;
    const long long row = strides != nullptr && t < n ? strides[2 * t + 1] : static_cast<long long>(H) * d;
    const bool kv = t == fa::kK || t == fa::kV || t == fa::kdK || t == fa::kdV;
    st[3 * t] = row * (kv ? total_k : total_q);  // one batch coordinate: the whole buffer
    st[3 * t + 1] = head;
    st[3 * t + 2] = row;
  }
  s = fa::check_strides(st, n);
  if (s != FA_OK) return s;
  *p = fa::Problem{B, H, max_q, d, causal ? 1 : 0, scale, 0, nullptr, {}};
  for (int t = 0; t < fa::kNumTensors; ++t) p->st[t] = fa::Strides{st[3 * t], st[3 * t + 1], st[3 * t + 2]};
  p->var = 1;
  p->Nk = max_k;
  p->cu_q = cu_q;
  p->cu_k = cu_k;
  p->rows_q = total_q;
  p->rows_k = total_k;
  p->max_q = max_q;
  p->max_k = max_k;
  return FA_OK;
}

// The device facts a Problem built from the arguments alone still lacks.
bool add_device(fa::Problem* p) {
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return false;
  p->num_sms = di.num_sms;
  p->status = di.status;
  return true;
}

fa_status var_fwd(fa::Problem p, const void* q, const void* k, const void* v, void* o,
                  float* lse, void* stream) {
  if (!add_device(&p)) return FA_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.cu_q != nullptr && fa::launch_varlen_check(p, st) != cudaSuccess) return FA_ERR_CUDA;
  return fa::launch_fwd(p, q, k, v, o, lse, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status var_bwd(fa::Problem p, const void* q, const void* k, const void* v,
                  const void* o, const float* lse, const void* dO, void* dq, void* dk, void* dv,
                  void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || !fa::aligned16(workspace) ||
      workspace_bytes <
          fa::bwd_var_workspace_bytes(p.cu_q != nullptr, p.B, p.H, p.rows_q, p.max_k, p.d))
    return FA_ERR_WORKSPACE;
  if (!add_device(&p)) return FA_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.cu_q != nullptr && fa::launch_varlen_check(p, st) != cudaSuccess) return FA_ERR_CUDA;
  return fa::launch_bwd(p, q, k, v, o, lse, dO, dq, dk, dv, workspace, fa::kStagesAll, st) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // namespace

fa_status fa_fwd_nqnk(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, const long long* strides, int causal,
                      float scale, void* stream) {
  fa::Problem p;
  fa_status s = nqnk_problem(&p, B, H, Nq, Nk, d, strides, 4, causal, scale);
  if (s != FA_OK) return s;
  s = fa::check_ptrs({q, k, v, o, lse});
  if (s != FA_OK) return s;
  return var_fwd(p, q, k, v, o, lse, stream);
}

fa_status fa_bwd_nqnk(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                      int H, int Nq, int Nk, int d, const long long* strides, int causal,
                      float scale, void* workspace, size_t workspace_bytes, void* stream) {
  fa::Problem p;
  fa_status s = nqnk_problem(&p, B, H, Nq, Nk, d, strides, fa::kNumTensors, causal, scale);
  if (s != FA_OK) return s;
  s = fa::check_ptrs({q, k, v, o, lse, dO, dq, dk, dv});
  if (s != FA_OK) return s;
  return var_bwd(p, q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, stream);
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                        const long long* strides, int causal, float scale, void* stream) {
  fa::Problem p;
  fa_status s = varlen_problem(&p, cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k,
                               max_seqlen_q, max_seqlen_k, d, strides, 4, causal, scale);
  if (s != FA_OK) return s;
  s = fa::check_ptrs({q, k, v, o, lse});
  if (s != FA_OK) return s;
  return var_fwd(p, q, k, v, o, lse, stream);
}

size_t fa_bwd_varlen_workspace_size(int B, int H, int total_q, int max_seqlen_k, int d) {
  if (fa::check_sizes(B, H, total_q, d, 1.f) != FA_OK || max_seqlen_k < 1) return 0;
  return fa::bwd_var_workspace_bytes(true, B, H, total_q, max_seqlen_k, d);
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                        const long long* strides, int causal, float scale, void* workspace,
                        size_t workspace_bytes, void* stream) {
  fa::Problem p;
  fa_status s = varlen_problem(&p, cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k,
                               max_seqlen_q, max_seqlen_k, d, strides, fa::kNumTensors, causal,
                               scale);
  if (s != FA_OK) return s;
  s = fa::check_ptrs({q, k, v, o, lse, dO, dq, dk, dv});
  if (s != FA_OK) return s;
  return var_bwd(p, q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, stream);
}

size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d) {
  if (fa::check_sizes(B, H, Nq, d, 1.f) != FA_OK || Nq > fa::kDecodeMaxQ || Nk < 1) return 0;
  // the plan depends on the SM count: the current device's, else the most
  // any plan can use (every split count up to kDecodeMaxSplits)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
    return std::max<size_t>(fa::decode_workspace_bytes(B, H, Nq, Nk, d, sms), 16);
  cudaGetLastError();  // no device here: clear the error
  int nqp = 1;
  while (nqp < Nq) nqp *= 2;
  const size_t splits = std::min((Nk + fa::kTile - 1) / fa::kTile, fa::kDecodeMaxSplits);
  return std::max<size_t>(static_cast<size_t>(B) * H * splits * nqp * (d + 1) * 4, 16);
}

fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    const int* cache_seqlens, int B, int H, int Nq, int Nk, int d,
                    const long long* strides, int causal, float scale, void* workspace,
                    size_t workspace_bytes, void* stream) {
  fa_status s = fa::check_sizes(B, H, Nq, d, scale);
  if (s != FA_OK) return s;
  if (Nq > fa::kDecodeMaxQ) return FA_ERR_UNSUPPORTED;
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  s = fa::check_ptrs({q, k_cache, v_cache, o, lse});
  if (s != FA_OK) return s;
  if (cache_seqlens != nullptr && (reinterpret_cast<uintptr_t>(cache_seqlens) & 3u) != 0)
    return FA_ERR_INVALID_ARG;
  if (strides != nullptr) {
    s = fa::check_strides(strides, 4);
    if (s != FA_OK) return s;
  }
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return FA_ERR_CUDA;
  const size_t need = fa::decode_workspace_bytes(B, H, Nq, Nk, d, di.num_sms);
  if (need > 0 && (workspace == nullptr || !fa::aligned16(workspace) || workspace_bytes < need))
    return FA_ERR_WORKSPACE;
  fa::Problem p{B, H, Nq, d, causal ? 1 : 0, scale, di.num_sms, di.status, {}};
  for (int t = 0; t < fa::kNumTensors; ++t) {
    const bool kv = t == fa::kK || t == fa::kV;
    p.st[t] = (strides != nullptr && t < 4)
                  ? fa::Strides{strides[3 * t], strides[3 * t + 1], strides[3 * t + 2]}
                  : fa::contiguous_strides(H, kv ? Nk : Nq, d);
  }
  p.Nk = Nk;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int tc_splits = fa::decode_tc_splits(B, H, Nk, di.num_sms);
  const bool fill = static_cast<int64_t>(B) * H >= di.num_sms;
  if (Nq >= fa::kDecodeTensorMinQ && (fill || (tc_splits > 1 && fa::fwd_split_supported(d)))) {
    // the tensor-core forward over a dense batch with per-sequence key
    // counts: over whole caches when the (batch, head) pairs fill the SMs,
    // else with the keys split by the decode plan and the splits merged by
    // log-sum-exp
    p.var = 1;
    p.rows_q = p.max_q = Nq;
    p.rows_k = p.max_k = Nk;
    p.cu_k = cache_seqlens;
    p.klens = cache_seqlens != nullptr;
    if (p.klens && fa::launch_klens_check(cache_seqlens, B, Nk, p.status, st) != cudaSuccess)
      return FA_ERR_CUDA;
    if (fill)
      return fa::launch_fwd(p, q, k_cache, v_cache, o, lse, st) == cudaSuccess ? FA_OK
                                                                              : FA_ERR_CUDA;
    float* part_o = static_cast<float*>(workspace);
    float* part_lse = part_o + static_cast<size_t>(B) * H * tc_splits * fa::nq_pad_of(Nq) * d;
    if (fa::launch_fwd_split(p, q, k_cache, v_cache, part_o, part_lse, tc_splits,
                             fa::nq_pad_of(Nq), st) != cudaSuccess)
      return FA_ERR_CUDA;
    return fa::launch_decode_combine(p, part_o, part_lse, tc_splits, o, lse, st) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
  }
  const cudaError_t e = fa::launch_decode(p, q, k_cache, v_cache, o, lse, cache_seqlens,
                                          workspace, st);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_measure_unit_rates(unsigned long long* cycles, int iters, void* stream) {
  if (cycles == nullptr || (reinterpret_cast<uintptr_t>(cycles) & 7u) != 0 || iters < 1 ||
      iters > (1 << 20))
    return FA_ERR_INVALID_ARG;
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return FA_ERR_CUDA;
  return fa::launch_unit_rates(cycles, iters, di.num_sms, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
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
  if (cudaMemcpyFromSymbol(&h, fa::g_device_word, sizeof(int), offsetof(fa::DeviceWord, status)) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  if (h != fa::DEV_OK) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_device_word, &zero, sizeof(int),
                           offsetof(fa::DeviceWord, status)) != cudaSuccess)
      return FA_ERR_CUDA;
    if (h == fa::DEV_BADARG) return FA_ERR_INVALID_ARG;
    return h == fa::DEV_BADINDEX ? FA_ERR_DEVICE_CHECK : FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

int fa_is_debug_build(void) {
#ifdef FA_DEBUG
  return 1;
#else
  return 0;
#endif
}

fa_status fa_set_wait_limit_ns(unsigned long long limit_ns) {
#ifndef FA_DEBUG
  (void)limit_ns;
  return FA_ERR_UNSUPPORTED;  // the release kernels keep the fixed limit
#else
  if (limit_ns > fa::kWaitLimitNs) return FA_ERR_INVALID_ARG;
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpyToSymbol(fa::g_device_word, &limit_ns, sizeof(limit_ns),
                         offsetof(fa::DeviceWord, wait_limit_ns)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
#endif
}

fa_status fa_selftest_index_check(void* stream) {
#ifndef FA_DEBUG
  (void)stream;
  return FA_ERR_UNSUPPORTED;  // the release build has no index checks
#else
  fa::DeviceInfo di;
  if (fa::device_info(&di) != cudaSuccess) return FA_ERR_CUDA;
  fa::index_check_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(di.status);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
#endif
}

}  // extern "C"

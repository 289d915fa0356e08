// Internal interface between the C ABI (fa_api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

constexpr int kTile = 128;  // query rows per Q tile and keys per K/V tile

// Element strides of one [B, H, N, d] tensor between batches, heads and rows;
// the d values of a row are contiguous.
struct Strides {
  int64_t batch, head, row;
};

// Tensors of a call, in this order in Problem::st.
enum TensorId : int { kQ = 0, kK, kV, kO, kdO, kdQ, kdK, kdV, kNumTensors };

// Everything a launcher needs besides the tensor pointers.
struct Problem {
  int B, H, N, d;
  int causal;
  float scale;
  int num_sms;
  int* status;  // device address of the status word
  Strides st[kNumTensors];
};

// Contiguous [B, H, N, d] strides.
inline Strides contiguous_strides(int H, int N, int d) {
  return Strides{static_cast<int64_t>(H) * N * d, static_cast<int64_t>(N) * d, d};
}

// Encodes a 4-D TMA map (d, N, H, B) over a bf16 tensor with the given
// strides, a {64, 128, 1, 1} box and 128-byte swizzle. Returns false on failure.
bool make_tile_map(CUtensorMap* map, const void* base, int B, int H, int N, int d,
                   const Strides& s);

// Launchers; they return a cudaError_t from the launch.
cudaError_t launch_fwd(const Problem& p, const void* q, const void* k, const void* v, void* o,
                       float* lse, cudaStream_t stream);

// The backward's three stages; pointers the stage does not use may be null.
enum BwdStage : int { kStagePre = 1, kStageDkdv = 2, kStageDq = 4, kStagesAll = 7 };

cudaError_t launch_bwd(const Problem& p, const void* q, const void* k, const void* v,
                       const void* o, const float* lse, const void* dO, void* dq, void* dk,
                       void* dv, void* workspace, int stages, cudaStream_t stream);

size_t bwd_workspace_bytes(int B, int H, int N, int d);

}  // namespace fa

// Internal interface between the C ABI (fa_api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
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
  // Sequences of unequal query and key lengths (var = 1), causal mask aligned
  // at the bottom right. Dense batch (cu_q null): B sequences of N query and
  // Nk key rows in [B, H, N | Nk, d] tensors. Packed batch: sequence b owns
  // rows cu_q[b]..cu_q[b+1]-1 of q and cu_k[b]..cu_k[b+1]-1 of k and v,
  // which hold rows_q and rows_k rows per head (batch coordinate 0); max_q
  // and max_k bound the lengths.
  int var = 0;
  int Nk = 0;
  const int* cu_q = nullptr;
  const int* cu_k = nullptr;  // dense batch with klens = 1: B valid key counts (see seq_of)
  int klens = 0;
  int rows_q = 0, rows_k = 0, max_q = 0, max_k = 0;
  // Backward of a dense batch: dQ by the query-stationary kernel (fa_bwd_dq.cu)
  // instead of atomics in the dK/dV kernel (d = 64 and 128).
  int dq_separate = 0;
};

// Debug build (FA_DEBUG): whether elements [off, off + n) of a [B, H, rows, d]
// tensor with these strides lie at or before its last element (and off >= 0).
// FA_IN_SPAN is that check in the debug build and true (arguments not
// evaluated) in the release build; kernels pass it to fa_dcheck (ptx.cuh).
#ifdef FA_DEBUG
__device__ __forceinline__ bool in_span(const Strides& st, int B, int H, int rows, int d,
                                        int64_t off, int n) {
  const int64_t last = static_cast<int64_t>(B - 1) * st.batch + static_cast<int64_t>(H - 1) * st.head +
                       static_cast<int64_t>(rows - 1) * st.row + d - 1;
  return off >= 0 && off + n - 1 <= last;
}
#define FA_IN_SPAN(st, B, H, rows, d, off, n) ::fa::in_span(st, B, H, rows, d, off, n)
#define FA_IN_RANGE(i, n) ((i) >= 0 && (i) < (n))
#else
#define FA_IN_SPAN(st, B, H, rows, d, off, n) true
#define FA_IN_RANGE(i, n) true
#endif

// Contiguous [B, H, N, d] strides.
inline Strides contiguous_strides(int H, int N, int d) {
  return Strides{static_cast<int64_t>(H) * N * d, static_cast<int64_t>(N) * d, d};
}

// Encodes a 4-D TMA map (d, N, H, B) over a bf16 tensor with the given
// strides, a {64, box_rows, 1, 1} box and 128-byte swizzle. Returns false on
// failure.
// box_blocks = 1: a 4-D map (d, row, head, batch) whose box is 64 columns by
// box_rows rows. box_blocks > 1 (d a multiple of 64): a 5-D map (64 columns,
// row, 64-column block, head, batch) whose box spans box_blocks blocks, for
// tma_load_5d.
bool make_tile_map(CUtensorMap* map, const void* base, int B, int H, int N, int d,
                   const Strides& s, int box_rows = kTile, int box_blocks = 1);

// scale * log2(e), at least 1e-30, for the kernels that turn masked scores
// into 2^-inf = 0 through their -inf value alone (the forwards), which needs
// a positive factor (-inf * 0 is NaN). At scale = 0
// the clamp changes the exponent of an unmasked score by |s| * 1e-30, i.e.
// nothing; the log-sum-exp keeps its max term from the true scale.
inline float clamped_scale_log2(float scale) {
  const float f = scale * 1.4426950408889634f;
  return f > 1e-30f ? f : 1e-30f;
}

// Launchers; they return a cudaError_t from the launch.

// The dK / dV stage at head dimension 256 (fa_bwd256.cu): its own kernel over
// 64-key blocks. The workspace rows are those of the d <= 128 backward:
// lse2 and D fp32 [BH, Npad] (Npad = N rounded up to 128; pad rows lse2 =
// +inf, D = 0) and the fp32 dQ accumulator [BH, N, 256].
struct Bwd256Args {
  const float* lse2;
  const float* Drow;
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  int N, H, Npad, BH, n_kb, n_qb, n_items;
  float scale, scale_log2;
  Strides sdk, sdv;
};
// maps: 5-D (make_tile_map with box_blocks = 4; q causal with 2), q and dO
// with 128-row boxes, k and v with 64-row boxes; a copy fills a whole tile
// (q causal: half a tile).
cudaError_t launch_bwd256_dkdv(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mdo,
                               const Bwd256Args& a, cudaStream_t stream);
// The separate dQ path (fa_bwd_dq.cu): one CTA per (batch*head, 128-row query
// block) recomputes S and dP against every key block it sees and accumulates
// dQ in TMEM; writes bf16 dq = scale * dQ directly. lse2 and D are the
// pre-pass rows [BH, Npad] of the d <= 128 backward.
struct BwdDqArgs {
  const float* lse2;
  const float* Drow;
  __nv_bfloat16* dq;
  int* status;
  int N, H, Npad, BH, n_tiles, n_items;
  float scale, scale_log2;
  Strides sdq;
};
bool bwd_dq_separate_supported(int d);
// maps: q, k, v, dO with 128-row boxes.
cudaError_t launch_bwd_dq_separate(const Problem& p, const CUtensorMap* maps, const BwdDqArgs& a,
                                   cudaStream_t stream);
cudaError_t launch_fwd(const Problem& p, const void* q, const void* k, const void* v, void* o,
                       float* lse, cudaStream_t stream);

// Forward at head dimension 256 (dense or strided [B, H, N, d], equal lengths).
cudaError_t launch_fwd256(const Problem& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, cudaStream_t stream);

// The backward's three stages; pointers the stage does not use may be null.
enum BwdStage : int { kStagePre = 1, kStageDkdv = 2, kStageDq = 4, kStagesAll = 7 };

cudaError_t launch_bwd(const Problem& p, const void* q, const void* k, const void* v,
                       const void* o, const float* lse, const void* dO, void* dq, void* dk,
                       void* dv, void* workspace, int stages, cudaStream_t stream);

size_t bwd_workspace_bytes(int B, int H, int N, int d);

// Decode: Nq <= kDecodeMaxQ new query rows per (batch, head) against a cache
// of up to Nk keys (cache_seqlens[b] of them when given), split along the
// keys over CTAs and merged by log-sum-exp.
constexpr int kDecodeMaxQ = 16;
// fa_decode runs N_q >= kDecodeTensorMinQ on the tensor-core forward for a
// dense batch with per-sequence key counts (no key split) once the B * H
// (batch, head) pairs fill the SMs. The split-key kernel below does its
// per-row arithmetic on CUDA cores: on GB300 (B = H = 32, 8192-key cache,
// d = 128) it read the cache at 7.1 / 6.9 / 5.4 / 3.2 / 1.4 TB/s for
// N_q = 1 / 2 / 4 / 8 / 16, the tensor-core forward at 5.2-5.4 TB/s for each
// (at N_q = 4 the two are within run-to-run noise).
constexpr int kDecodeTensorMinQ = 8;
constexpr int kDecodeMaxSplits = 256;

struct DecodePlan {
  int splits;           // key splits per (batch, head)
  int tiles_per_split;  // 128-key tiles per split
};

DecodePlan decode_plan(int B, int H, int Nk, int num_sms);
size_t decode_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_sms);

// Decode on the tensor-core forward with the keys split (d = 64 and 128): a
// dense batch (p.var, p.cu_q null, p.klens as for the forward) of Nq <= 128
// query rows per sequence; item (b*h, split s) covers an even share of the
// key tiles the sequence's rows see and writes its normalised rows and log2
// LSE to part_o [B*H, splits, nq_pad, d] and part_lse [B*H, splits, nq_pad]
// (splits past the keys: 0 and -inf). launch_decode_combine merges.
bool fwd_split_supported(int d);
// Splits per (batch, head) for it: the fewest from ceil(SMs / (B*H)) up
// whose B*H*splits work items fill their rounds of one item per SM to 95%
// (the persistent grid takes several rounds), at most one per key tile.
int decode_tc_splits(int B, int H, int Nk, int num_sms);
cudaError_t launch_fwd_split(const Problem& p, const void* q, const void* k, const void* v,
                             float* part_o, float* part_lse, int splits, int nq_pad,
                             cudaStream_t stream);
// O = sum_s 2^(lse_s - lse) O_s over the splits, into o (p.st[kO]) and lse.
cudaError_t launch_decode_combine(const Problem& p, const float* part_o, const float* part_lse,
                                  int splits, void* o, float* lse, cudaStream_t stream);
int nq_pad_of(int Nq);

// p.N = Nq, p.Nk = Nk; p.st holds the strides of q, k, v, o (kQ .. kO).
cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, const int* cache_seqlens, void* workspace,
                          cudaStream_t stream);

// Workspace of the backward for unequal lengths (packed = false: B dense
// sequences of rows_q query rows) or a packed batch of B sequences with
// rows_q query rows in all: D and the log2 LSE rows (fp32) padded per
// sequence, then the fp32 dQ accumulator (and, packed, the compacted work
// schedule, sized by the longest key sequence max_k).
size_t bwd_var_workspace_bytes(bool packed, int B, int H, int rows_q, int max_k, int d);

// The arithmetic-unit microbenchmark (fa_unit_rates.cu): writes the largest
// block cycle count of the ex2, FFMA and FFMA2 kernels to cycles[0], [2], [4].
cudaError_t launch_unit_rates(unsigned long long* cycles, int iters, int num_sms,
                              cudaStream_t stream);

// Records DEV_BADARG in the status word when one of the B key counts is
// outside 0..Nk.
cudaError_t launch_klens_check(const int* lens, int B, int Nk, int* status, cudaStream_t stream);

// Records DEV_BADARG in the status word when the packed batch's offsets are
// not non-decreasing from 0 to rows_q / rows_k or a length exceeds max_q /
// max_k. The kernels clamp every offset, so such offsets give wrong results
// but no access outside the buffers.
cudaError_t launch_varlen_check(const Problem& p, cudaStream_t stream);

}  // namespace fa

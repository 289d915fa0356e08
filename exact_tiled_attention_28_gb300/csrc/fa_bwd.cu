// Backward kernels: recompute S and P per tile, then dP, dS, dV, dK, dQ.
//
// What it computes ("Flash Attention v2" notes, "Backward Pass Computation":
// recompute S block by block from Q and K, then the gradients block by
// block, never materialising N x N matrices; the softmax Jacobian is the full
// one, not the diagonal form printed there):
//   D_i = sum_c dO_ic O_ic                       (pre-pass)
//   P_ij = exp(scale q_i.k_j - lse_i)            (recomputed from the forward's lse)
//   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i)
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K
//
// GB300 mapping:
//  1. bwd_pre_kernel (memory bound): D, the log-sum-exp in log2 units, both
//     padded to whole 128-row tiles (pad rows: D = 0, lse2 = +inf so that P
//     vanishes there), and zeroes the fp32 dQ accumulator.
//  2. bwd_dkdv_kernel: persistent CTAs over (batch*head, key block j). A CTA
//     keeps K_j and V_j in shared memory and dV_j, dK_j in tensor memory and
//     loops over the query blocks i (causal: i >= j, longest blocks first):
//       S^T = K_j Q_i^T and dP^T = V_j dO_i^T       (tcgen05, SS)
//       P^T, dS^T by two compute warpgroups, one thread per key row, each
//       warpgroup owning 64 of the 128 query columns  (TMEM -> regs; P^T
//       back to TMEM, dS^T to swizzled shared memory)
//       dV += P^T dO_i                              (tcgen05, A from TMEM)
//       d >= 64: dQ_i^T = K_j^T dS^T (M = 128)      (tcgen05, both from SMEM)
//       d = 32:  dQ_i = dS K_j                      (tcgen05, both from SMEM)
//       dK += dS^T Q_i                              (tcgen05, both from SMEM)
//     and four more warps read dQ_i out of TMEM and add it to the fp32
//     accumulator in global memory. With dQ^T in TMEM (lanes = head dim,
//     columns = queries) a warp's 32 atomics cover one contiguous 128-byte
//     row segment.
//  3. dq_convert_kernel: dq = bf16(scale * accumulator).
//
// TMEM (512 columns): S^T [0,128), dP^T then dQ_i [128,256), dV [256, 256+d),
// dK [256+d, 256+2d). Compute warpgroup c reads columns 64c..64c+63 of S^T and
// dP^T and writes its packed bf16 P^T (two per column) over the first 32 of
// its S^T columns, so neither warpgroup overwrites a column the other still
// has to read; the dV MMA addresses the two 32-column halves separately.
// MMA order per query block, non-causal: dV(i), S^T(i+1), dQ(i), dK(i),
// dP^T(i+1), with dK reading dS^T from shared memory: dQ_i comes before dK so
// that its read-out from the dP^T columns overlaps the dK product (dP^T(i+1)
// waits for that read-out). Causal: dV(i), S^T(i+1), dK(i), dQ(i), dP^T(i+1)
// with dK reading dS^T from TMEM (the compute warps also store it there);
// each order measured faster for its case on GB300 (by about 2.5%). At
// d = 64 non-causal: dV(i), dK(i) from TMEM, dQ(i), S^T(i+1), dP^T(i+1)
// (3% faster there; 13% slower at d = 128).

#include <algorithm>

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "schedule.cuh"
#include "seq.cuh"

namespace fa {
namespace {

// four warpgroups: 0-1 compute, 2 dQ readout, 3 = load warp, MMA warp, two idle
constexpr int kBwdThreads = 512;
constexpr int kBwdDqWarp0 = 8;
constexpr int kBwdLoadWarp = 12;
constexpr int kBwdMmaWarp = 13;
constexpr uint32_t kBwdTmemCols = 512;
constexpr int kBlk = kTile * 64 * 2;  // 16 KiB: one 128-row x 64-column bf16 block
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256;
constexpr int kSmemSpare = 768;  // bytes left for aligning the dynamic base to 1024

template <int D>
struct BwdCfg {
  // d = 32 and 96 use whole 64-column blocks (TMA zero-fills past d)
  static constexpr int kColBlocks = (D + 63) / 64;
  static constexpr int kTileBytes = kTile * kColBlocks * 64 * 2;
  static constexpr int kStages = 2;
  static constexpr int kStageBytes = 2 * kTileBytes + 1024;  // Q_i, dO_i, lse2 and D rows
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffDS = 2 * kTileBytes;             // dS^T, 128 x 128 bf16
  static constexpr int kOffStages = 2 * kTileBytes + kTile * kTile * 2;
  // d = 64: a second copy of K_j, the second 64-row half of the dQ_i^T
  // product's A operand, so that all 128 TMEM lanes of dQ_i^T hold real
  // values (rows 64-127 repeat rows 0-63) and all four dQ warps share the
  // read-out and its atomics, half of the query columns each. With rows
  // 64-127 unused, two warps issued every atomic: on GB300 those took about
  // 3900 of the 4750 cycles of a query block.
  static constexpr bool kDupK = D == 64;
  static constexpr int kOffK2 = kOffStages + kStages * kStageBytes;
  static constexpr int kOffBars = kOffK2 + (kDupK ? kTileBytes : 0);
  // d >= 64: dQ_i^T = K^T dS^T with M = 128, read out with coalesced atomics.
  // At d = 96 the MMA's rows past d read the K tile's zero-filled columns and
  // are never stored; at d = 64 they read the copy of K (kDupK). Measured on
  // GB300 at d = 64, with rows 64-127 unused, this beat dQ_i = dS K with one
  // scattered row per thread by 22%.
  // d = 32: dQ_i = dS K with one row per thread.
  static constexpr bool kDqTransposed = D >= 64;
  static constexpr uint32_t col_dk() { return kColDV + D; }
};

struct BwdBarriers {
  uint64_t kv_full, kv_empty;
  uint64_t st_full[2], st_empty[2];
  uint64_t s_full, dp_full, p_ready, ds_ready, dq_full, dq_free, acc_done, drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
constexpr int bwd_smem_bytes() {
  return BwdCfg<D>::kOffBars + static_cast<int>(sizeof(BwdBarriers)) + kSmemSpare;
}
static_assert(bwd_smem_bytes<128>() <= 232448, "backward shared memory over the sm_103a limit");
static_assert(bwd_smem_bytes<64>() <= 232448, "backward shared memory over the sm_103a limit");
static_assert(bwd_smem_bytes<96>() <= 232448, "backward shared memory over the sm_103a limit");

// The workspace: D and the lse rows in log2 units, each fp32 [BH, Npad], then
// the fp32 dQ accumulator [BH, N, d].
// (Host code reads the same offsets to hand them to the d = 256 kernel.)
struct Workspace {
  float* base;
  __host__ __device__ __forceinline__ float* Drow(int BH, int Npad) const { return base; }
  __host__ __device__ __forceinline__ float* lse2(int BH, int Npad) const {
    return base + static_cast<size_t>(BH) * Npad;
  }
  __host__ __device__ __forceinline__ float* dq_acc(int BH, int Npad) const {
    return base + 2 * static_cast<size_t>(BH) * Npad;
  }
};

// Each kernel gets only the arguments it reads. The dK/dV kernel's struct is
// kept at 112 bytes: with more (even unused) bytes appended, its launches ran
// 3-12% slower on GB300 with this compiler.
struct PreArgs {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dO;
  const float* lse;
  Workspace ws;
  Strides so, sdo;  // element strides of o and dO
  int N, H, Npad, BH;
  int zero_acc;  // zero the fp32 dQ accumulator (the atomic dQ path only)
};

struct DqArgs {
  Workspace ws;
  __nv_bfloat16* dq;
  Strides sdq;
  int N, H, Npad, BH;
  float scale;
  int* status;  // debug build: index checks
};

struct BwdArgs {
  Workspace ws;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  int N, H, Npad, BH, n_tiles, n_items;
  float scale, scale_log2;
  Strides sdk, sdv;  // element strides of dk and dv
};
static_assert(sizeof(BwdArgs) == 112, "dK/dV argument struct grew");

// Sequences of unequal lengths (dense or packed batch; sh = b * H + h runs
// over sequences and heads). The workspace holds D and lse2 as
// [planes, lpad] (each sequence's rows from its Seq::pst on, whole 128-row
// tiles, pad rows D = 0 and lse2 = +inf), then the fp32 accumulator
// [planes, rows_q, d]; planes = batch coordinates x H.
struct PreVarArgs {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dO;
  const float* lse;  // [planes, rows_q]
  float* ws;
  Strides so, sdo;
  int planes, lpad, max_q_pad, BH;
  VarGeom g;
};

struct BwdVarArgs {
  float* ws;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  int BH, n_tiles, n_items;  // n_tiles: key tiles of the longest sequence
  int planes, lpad;
  float scale, scale_log2;
  Strides sdk, sdv;
  VarGeom g;
  // packed batch: the compacted, longest-first schedule (seq.cuh, Sched) in
  // the workspace, written by bwd_var_sched_kernel; levels = key tiles,
  // causal visited from 0 (the most query blocks). Null for a dense batch.
  int* sched;
  int n_seq, sched_P;
};

// The compacted schedule of a packed batch (one block): every sequence with
// keys owns its key tiles as levels, also when it has no queries (those items
// zero its dK and dV).
template <bool CAUSAL>
__global__ void __launch_bounds__(kSchedBuildThreads) bwd_var_sched_kernel(VarGeom g, int n_seq,
                                                                           int P, int* base) {
  build_sched(sched_arrays(base, n_seq, P), n_seq, P, g.H, CAUSAL, /*top_first=*/false,
              [&](int b) { return (seq_of(b * g.H, g).nk + kTile - 1) / kTile; },
              base + sched_ints(n_seq, P), static_cast<int>(sched_build_scratch_ints(P)));
}

template <bool VAR>
struct BwdArgsOf {
  using type = BwdArgs;
};
template <>
struct BwdArgsOf<true> {
  using type = BwdVarArgs;
};

// Element offset of row `row` of head bh (= b * H + h) in a strided tensor.
__device__ __forceinline__ int64_t row_offset(const Strides& st, int bh, int H, int row) {
  return (bh / H) * st.batch + (bh % H) * st.head + static_cast<int64_t>(row) * st.row;
}

// ---------------------------------------------------------------------------
// 1. pre-pass

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreArgs a) {
  // each active lane handles 8 elements (16 bytes) of a row; rows take a
  // power-of-two number of lanes, the ones past d / 8 idle (d = 96)
  constexpr int kLanesPerRow = D <= 32 ? 4 : (D <= 64 ? 8 : (D <= 128 ? 16 : 32));
  constexpr int kActive = D / 8;
  const size_t rows = static_cast<size_t>(a.BH) * a.Npad;
  float* const Drow = a.ws.Drow(a.BH, a.Npad);
  float* const lse2 = a.ws.lse2(a.BH, a.Npad);
  float* const dq_acc = a.ws.dq_acc(a.BH, a.Npad);
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t g = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       g < rows * kLanesPerRow; g += nthreads) {
    const size_t row = g / kLanesPerRow;
    const int part = static_cast<int>(g % kLanesPerRow);
    const int bh = static_cast<int>(row / a.Npad);
    const int i = static_cast<int>(row % a.Npad);
    float dot = 0.f;
    if (i < a.N && part < kActive) {
      const size_t e = (static_cast<size_t>(bh) * a.N + i) * D + part * 8;  // accumulator
      const uint4 ov = *reinterpret_cast<const uint4*>(a.o + row_offset(a.so, bh, a.H, i) + part * 8);
      const uint4 gv =
          *reinterpret_cast<const uint4*>(a.dO + row_offset(a.sdo, bh, a.H, i) + part * 8);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 of = __bfloat1622float2(o2[u]);
        const float2 gf = __bfloat1622float2(g2[u]);
        dot = fmaf(of.x, gf.x, dot);
        dot = fmaf(of.y, gf.y, dot);
      }
      if (a.zero_acc) {
        float4* z = reinterpret_cast<float4*>(dq_acc + e);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    // reduce over the kLanesPerRow consecutive lanes of this row
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
      dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (part == 0) {
      Drow[row] = dot;
      lse2[row] = (i < a.N) ? a.lse[static_cast<size_t>(bh) * a.N + i] * 1.4426950408889634f
                              : __int_as_float(0x7f800000);
    }
  }
}

// The pre-pass for sequences of unequal lengths: one unit per (sequence,
// head, row r < roundup(max_q, 128)); rows past the sequence's padded length
// do nothing. A row whose forward saw no key (LSE = -inf) gets lse2 = +inf,
// so that its P is 0 and it adds nothing to any gradient.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_var_kernel(const PreVarArgs a) {
  constexpr int kLanesPerRow = D <= 32 ? 4 : (D <= 64 ? 8 : (D <= 128 ? 16 : 32));
  constexpr int kActive = D / 8;
  const size_t units = static_cast<size_t>(a.BH) * a.max_q_pad;
  float* const Drow = a.ws;
  float* const lse2 = a.ws + static_cast<size_t>(a.planes) * a.lpad;
  float* const dq_acc = a.ws + 2 * static_cast<size_t>(a.planes) * a.lpad;
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t g = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       g < units * kLanesPerRow; g += nthreads) {
    const size_t unit = g / kLanesPerRow;
    const int part = static_cast<int>(g % kLanesPerRow);
    const int sh = static_cast<int>(unit / a.max_q_pad);
    const int r = static_cast<int>(unit % a.max_q_pad);
    const Seq sq = seq_of(sh, a.g);
    const size_t plane = static_cast<size_t>(sq.bb) * a.g.H + sq.hh;
    const bool real = r < sq.nq;
    const bool padded = r < (sq.nq + kTile - 1) / kTile * kTile;
    float dot = 0.f;
    if (real && part < kActive) {
      const int64_t row = sq.q0 + r;
      const uint4 ov = *reinterpret_cast<const uint4*>(a.o + sq.bb * a.so.batch + sq.hh * a.so.head +
                                                       row * a.so.row + part * 8);
      const uint4 gv = *reinterpret_cast<const uint4*>(
          a.dO + sq.bb * a.sdo.batch + sq.hh * a.sdo.head + row * a.sdo.row + part * 8);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 of = __bfloat1622float2(o2[u]);
        const float2 gf = __bfloat1622float2(g2[u]);
        dot = fmaf(of.x, gf.x, dot);
        dot = fmaf(of.y, gf.y, dot);
      }
      float4* z = reinterpret_cast<float4*>(dq_acc + (plane * a.g.rows_q + row) * D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
      dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (part == 0 && padded) {
      const size_t idx = plane * a.lpad + sq.pst + r;
      float l2 = __int_as_float(0x7f800000);
      if (real) {
        const float lse = a.lse[plane * a.g.rows_q + sq.q0 + r];
        if (lse != __int_as_float(0xff800000)) l2 = lse * 1.4426950408889634f;
      }
      Drow[idx] = dot;
      lse2[idx] = l2;
    }
  }
}

// ---------------------------------------------------------------------------
// 3. dq = bf16(scale * accumulator)

template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const DqArgs a, size_t n8) {
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t g = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < n8;
       g += nthreads) {
    const float4* src = reinterpret_cast<const float4*>(a.ws.dq_acc(a.BH, a.Npad)) + 2 * g;
    const float4 x = src[0], y = src[1];
    const size_t row = g / (D / 8);  // accumulator row (b*H + h) * N + i
    const int col = static_cast<int>(g % (D / 8)) * 8;
    const int bh = static_cast<int>(row / a.N), i = static_cast<int>(row % a.N);
    if (!fa_dcheck(FA_IN_SPAN(a.sdq, a.BH / a.H, a.H, a.N, D, row_offset(a.sdq, bh, a.H, i) + col, 8),
                   a.status))
      continue;
    uint4 w;
    w.x = pack_bf16x2(x.x * a.scale, x.y * a.scale);
    w.y = pack_bf16x2(x.z * a.scale, x.w * a.scale);
    w.z = pack_bf16x2(y.x * a.scale, y.y * a.scale);
    w.w = pack_bf16x2(y.z * a.scale, y.w * a.scale);
    *reinterpret_cast<uint4*>(a.dq + row_offset(a.sdq, bh, a.H, i) + col) = w;
  }
}

// ---------------------------------------------------------------------------
// 2. dK / dV (and dQ contributions)

template <class Args>
__device__ __forceinline__ void decode_kv_item(int item, const Args& a, bool causal, int& bh,
                                               int& j) {
  if (causal) {  // key block 0 visits every query block: longest first
    j = item / a.BH;
    bh = item % a.BH;
  } else {  // blocks of one head adjacent: Q and dO shared through L2
    bh = item / a.n_tiles;
    j = item % a.n_tiles;
  }
}

// The u-th query block visited by key block j. Causal: j, j+1, ..., n_q-1.
// Non-causal: all blocks, starting at j and wrapping around, so that the CTAs
// working on neighbouring key blocks of one head at the same time add into
// different dQ rows instead of contending for the same ones.
__device__ __forceinline__ int qblock_at(int j, int u, int n_q, bool causal) {
  if (causal) return j + u;
  const int i = j + u;
  return i < n_q ? i : i - n_q;
}

// Query blocks that key block j of a sequence of unequal lengths visits:
// causal, the blocks from the first one holding a query that sees key
// j * 128 (bottom-right alignment) to the last; otherwise all of them,
// starting at j mod n_q. n_it = 0 when the key block lies past the sequence
// or the sequence has no queries.
struct KvWork {
  int n_it, i0, rot, n_q;
};

__device__ __forceinline__ KvWork var_kv_work(int j, const Seq& sq, bool causal) {
  KvWork w{0, 0, 0, 0};
  if (sq.nq <= 0 || j * kTile >= sq.nk) return w;
  w.n_q = (sq.nq + kTile - 1) / kTile;
  if (causal) {
    const int first = j * kTile - (sq.nk - sq.nq);
    w.i0 = first > 0 ? first / kTile : 0;
    w.n_it = w.n_q - w.i0;
  } else {
    w.rot = j % w.n_q;
    w.n_it = w.n_q;
  }
  return w;
}

__device__ __forceinline__ int var_qblock(const KvWork& w, int u, bool causal) {
  if (causal) return w.i0 + u;
  const int i = w.rot + u;
  return i < w.n_q ? i : i - w.n_q;
}

// 512 threads at 128 registers fill the register file (each SM sub-partition
// holds one warp of every warpgroup: 4 x 32 x 128 = 16384). The warpgroups then
// rebalance with setmaxnreg: compute 128, dQ readout 176, load/MMA 80; per
// sub-partition 128 + 128 + 176 + 80 = 512 registers per lane, the launch total.
// DQ = false (the separate dQ path, fa_bwd_dq.cu): no dQ product and no
// read-out; dS^T stays in TMEM only and both dK orders read it there, as
// dV(i), S^T(i+1), dK(i), dP^T(i+1).
template <int D, bool CAUSAL, bool VAR, bool DQ = true>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const typename BwdArgsOf<VAR>::type a) {
  using Cfg = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  const uintptr_t aligned = (raw + 1023) & ~static_cast<uintptr_t>(1023);
  if (aligned - raw > kSmemSpare) {  // cannot happen with a 1 KiB-aligned dynamic base
    if (threadIdx.x == 0) atomicCAS(a.status, DEV_OK, DEV_TIMEOUT);
    return;
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>(aligned);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + Cfg::kOffK, sV = sbase + Cfg::kOffV, sDS = sbase + Cfg::kOffDS;
  const uint32_t sSt = sbase + Cfg::kOffStages;
  const uint32_t sK2 = sbase + Cfg::kOffK2;
  BwdBarriers* bars = reinterpret_cast<BwdBarriers*>(smem + Cfg::kOffBars);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_q = a.n_tiles;  // VAR: key tiles of the longest sequence (unused as query blocks)

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->kv_full), 1);
    mbar_init(smem_u32(&bars->kv_empty), 1);
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(smem_u32(&bars->st_full[s]), 1);
      mbar_init(smem_u32(&bars->st_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->dp_full), 1);
    mbar_init(smem_u32(&bars->p_ready), 8);   // one elected lane per compute warp
    mbar_init(smem_u32(&bars->ds_ready), 8);
    mbar_init(smem_u32(&bars->dq_full), 1);
    mbar_init(smem_u32(&bars->dq_free), 4);   // one elected lane per dQ warp
    mbar_init(smem_u32(&bars->acc_done), 1);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kBwdTmemCols);
    tmem_relinquish();
  }
  if (warp == kBwdLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int n_eff = a.n_items;  // items of the schedule
  if constexpr (VAR) {
    if (a.sched != nullptr)
      n_eff = sched_total(sched_arrays(a.sched, a.n_seq, a.sched_P), a.n_seq, a.sched_P, CAUSAL);
  }

  if (warp >= kBwdLoadWarp) {
    setmaxnreg_dec<80>();
  if (warp == kBwdLoadWarp) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      uint32_t st_it = 0, kv_round = 0;
      bool ok = true;
      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= n_eff) break;  // only in the last, partial round
        int bh, j;
        if constexpr (VAR) {
          if (a.sched != nullptr) {
            int b, h;
            sched_decode(sched_arrays(a.sched, a.n_seq, a.sched_P), a.n_seq, a.sched_P, a.g.H,
                         CAUSAL, false, item, b, h, j);
            bh = b * a.g.H + h;
          } else {
            decode_kv_item(item, a, CAUSAL, bh, j);
          }
        } else {
          decode_kv_item(item, a, CAUSAL, bh, j);
        }
        int hh, bb, q0 = 0, k0 = 0, n_it;
        KvWork w;
        size_t lrow = 0;  // VAR: first padded D / lse2 row of the sequence
        if constexpr (VAR) {
          const Seq sq = seq_of(bh, a.g);
          w = var_kv_work(j, sq, CAUSAL);
          if (w.n_it == 0) continue;
          hh = sq.hh;
          bb = sq.bb;
          q0 = sq.q0;
          k0 = sq.k0;
          n_it = w.n_it;
          lrow = (static_cast<size_t>(sq.bb) * a.g.H + sq.hh) * a.lpad + sq.pst;
        } else {
          hh = bh % a.H;
          bb = bh / a.H;
          n_it = CAUSAL ? n_q - j : n_q;
        }
        auto load_stage = [&](int u) {
          int i;
          if constexpr (VAR)
            i = var_qblock(w, u, CAUSAL);
          else
            i = qblock_at(j, u, n_q, CAUSAL);
          const uint32_t s = st_it % Cfg::kStages;
          ok = mbar_wait(smem_u32(&bars->st_empty[s]), ((st_it / Cfg::kStages) & 1) ^ 1, abort,
                         a.status);
          if (!ok) return;
          const uint32_t bar = smem_u32(&bars->st_full[s]);
          const uint32_t st = sSt + s * Cfg::kStageBytes;
          mbar_arrive_expect_tx(bar, 2 * Cfg::kTileBytes + 1024);
          for (int cb = 0; cb < Cfg::kColBlocks; ++cb) {
            tma_load_4d(st + cb * kBlk, &tmQ, bar, 64 * cb, q0 + i * kTile, hh, bb, pol_q);
            tma_load_4d(st + Cfg::kTileBytes + cb * kBlk, &tmdO, bar, 64 * cb, q0 + i * kTile, hh,
                        bb, pol_q);
          }
          if constexpr (VAR) {
            const size_t roff = lrow + static_cast<size_t>(i) * kTile;
            const size_t plane_rows = static_cast<size_t>(a.planes) * a.lpad;
            cp_bulk_g2s(st + 2 * Cfg::kTileBytes, a.ws + plane_rows + roff, 512, bar);
            cp_bulk_g2s(st + 2 * Cfg::kTileBytes + 512, a.ws + roff, 512, bar);
          } else {
            const size_t roff = static_cast<size_t>(bh) * a.Npad + static_cast<size_t>(i) * kTile;
            cp_bulk_g2s(st + 2 * Cfg::kTileBytes, a.ws.lse2(a.BH, a.Npad) + roff, 512, bar);
            cp_bulk_g2s(st + 2 * Cfg::kTileBytes + 512, a.ws.Drow(a.BH, a.Npad) + roff, 512, bar);
          }
          ++st_it;
        };
        // dense batches: the first query block's stage goes out before the
        // wait for the K/V buffer, which frees only when the previous item's
        // last MMAs are done. Issued after it, the stage arrived about 2300
        // cycles after K and V at a causal d = 128 item boundary on GB300; the
        // early stage made the dK/dV kernel 0.5-0.7% faster at d = 64 and at
        // causal d = 128, and the packed d = 64 batch 1% slower.
        if constexpr (!VAR) {
          load_stage(0);
          if (!ok) break;
        }
        ok = mbar_wait(smem_u32(&bars->kv_empty), (kv_round & 1) ^ 1, abort, a.status);
        if (!ok) break;
        {
          const uint32_t bar = smem_u32(&bars->kv_full);
          constexpr bool kDup = DQ && Cfg::kDupK;
          mbar_arrive_expect_tx(bar, (kDup ? 3 : 2) * Cfg::kTileBytes);
          for (int cb = 0; cb < Cfg::kColBlocks; ++cb) {
            tma_load_4d(sK + cb * kBlk, &tmK, bar, 64 * cb, k0 + j * kTile, hh, bb, pol_kv);
            tma_load_4d(sV + cb * kBlk, &tmV, bar, 64 * cb, k0 + j * kTile, hh, bb, pol_kv);
          }
          if constexpr (kDup) tma_load_4d(sK2, &tmK, bar, 0, k0 + j * kTile, hh, bb, pol_kv);
          ++kv_round;
        }
        for (int u = VAR ? 0 : 1; u < n_it && ok; ++u) load_stage(u);
      }
      // producer tail (see the forward kernel)
      const uint32_t n = min(st_it, static_cast<uint32_t>(Cfg::kStages));
      for (uint32_t u = st_it - n; u < st_it; ++u) {
        const uint32_t s = u % Cfg::kStages, ph = (u / Cfg::kStages) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->st_empty[s]), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->st_full[s]), ph, 100000000ull);
      }
      if (kv_round > 0) {
        const uint32_t ph = (kv_round - 1) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->kv_empty), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->kv_full), ph, 100000000ull);
      }
    }
  } else if (warp == kBwdMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // S^T = K Q^T, dP^T = V dO^T: M = 128 keys, N = 128 queries, K-major operands
      constexpr uint32_t idesc_kq = idesc_bf16_f32(kTile, kTile, false, false);
      // dV += P^T dO, dK += dS^T Q: A from TMEM, B MN-major, N = d
      constexpr uint32_t idesc_acc = idesc_bf16_f32(kTile, D, false, true);
      // d = 128: dQ^T = K^T dS^T (M = d, N = 128 queries); d = 64: dQ = dS K
      // (M = 128 queries, N = d). Both operands MN-major in SMEM.
      constexpr uint32_t idesc_dq =
          idesc_bf16_f32(kTile, Cfg::kDqTransposed ? kTile : D, true, true);
      uint32_t st_it = 0, kv_round = 0, it = 0;
      bool ok = true;

      // Descriptors are rebuilt at every issue from an opaque base (one add per
      // K step): hoisted out of the loops they would not fit in the 80
      // registers of this warpgroup and would spill.
      auto issue_kq = [&](uint32_t dst, uint32_t a_tile, uint32_t b_tile) {
        const SmemDesc da = make_desc_sw128(opaque_u32(a_tile), 16, 1024);
        const SmemDesc db = make_desc_sw128(opaque_u32(b_tile), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
          mma_ss(dst, desc_at(da, off), desc_at(db, off), idesc_kq, kk > 0);
        }
      };
      // A = packed P^T or dS^T: queries 16kk..16kk+15 sit in the half of the
      // region written by compute warpgroup kk / 4, at column 64 (kk/4) + 8 (kk%4)
      auto issue_acc = [&](uint32_t dst, uint32_t a_region, uint32_t b_tile, bool accumulate) {
        const SmemDesc db = make_desc_sw128(opaque_u32(b_tile), kBlk, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(dst, a_region + 64 * (kk >> 2) + 8 * (kk & 3), desc_at(db, kk * 2048), idesc_acc,
                 (accumulate || kk > 0) ? 1u : 0u);
      };
      // dK += dS^T Q: A = dS^T from shared memory (keys x queries, K-major,
      // the buffer the dQ product reads too), B = Q_i MN-major. Reading dS^T
      // from shared memory rather than TMEM frees the dP^T columns for dQ_i
      // before dK is issued, so the dQ read-out overlaps the dK product.
      auto issue_dk = [&](uint32_t q_tile, bool accumulate) {
        const SmemDesc da = make_desc_sw128(opaque_u32(sDS), 16, 1024);
        const SmemDesc db = make_desc_sw128(opaque_u32(q_tile), kBlk, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ss(tmem + Cfg::col_dk(), desc_at(da, (kk >> 2) * kBlk + (kk & 3) * 32),
                 desc_at(db, kk * 2048), idesc_acc, (accumulate || kk > 0) ? 1u : 0u);
      };
      auto issue_dq = [&]() {
        const SmemDesc d_ds = make_desc_sw128(opaque_u32(sDS), kBlk, 1024);
        const SmemDesc d_kmn =
            make_desc_sw128(opaque_u32(sK), Cfg::kDupK ? sK2 - sK : kBlk, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t ds_desc = desc_at(d_ds, kk * 2048);
          const uint64_t k_desc = desc_at(d_kmn, kk * 2048);
          if constexpr (Cfg::kDqTransposed)
            mma_ss(tmem + kColDP, k_desc, ds_desc, idesc_dq, kk > 0);
          else
            mma_ss(tmem + kColDP, ds_desc, k_desc, idesc_dq, kk > 0);
        }
      };

      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd, ++kv_round) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= n_eff) break;  // only in the last, partial round
        int bh, j;
        if constexpr (VAR) {
          if (a.sched != nullptr) {
            int b, h;
            sched_decode(sched_arrays(a.sched, a.n_seq, a.sched_P), a.n_seq, a.sched_P, a.g.H,
                         CAUSAL, false, item, b, h, j);
            bh = b * a.g.H + h;
          } else {
            decode_kv_item(item, a, CAUSAL, bh, j);
          }
        } else {
          decode_kv_item(item, a, CAUSAL, bh, j);
        }
        int n_it;
        if constexpr (VAR) {
          n_it = var_kv_work(j, seq_of(bh, a.g), CAUSAL).n_it;
          if (n_it == 0) {  // skipped by the loader too: no K/V round
            --kv_round;
            continue;
          }
        } else {
          n_it = n_q - (CAUSAL ? j : 0);
        }
        ok = mbar_wait(smem_u32(&bars->kv_full), kv_round & 1, abort, a.status);
        if (!ok) break;
        // prologue: S^T(0), dP^T(0); dP needs the dQ readout of the previous item done
        uint32_t s0 = st_it % Cfg::kStages;
        ok = mbar_wait(smem_u32(&bars->st_full[s0]), (st_it / Cfg::kStages) & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t stq = sSt + s0 * Cfg::kStageBytes;
        issue_kq(tmem + kColS, sK, stq);
        mma_commit(smem_u32(&bars->s_full));
        if (DQ && it > 0) {
          ok = mbar_wait(smem_u32(&bars->dq_free), (it - 1) & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
        }
        issue_kq(tmem + kColDP, sV, stq + Cfg::kTileBytes);
        mma_commit(smem_u32(&bars->dp_full));
        for (int u = 0; u < n_it && ok; ++u, ++it, ++st_it) {
          const uint32_t s = st_it % Cfg::kStages;
          const uint32_t stage = sSt + s * Cfg::kStageBytes;
          const bool has_next = u + 1 < n_it;
          const uint32_t sn = (st_it + 1) % Cfg::kStages;
          const uint32_t next = sSt + sn * Cfg::kStageBytes;
          ok = mbar_wait(smem_u32(&bars->p_ready), it & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
          issue_acc(tmem + kColDV, tmem + kColS, stage + Cfg::kTileBytes, u > 0);  // dV += P^T dO
          if (has_next) {
            ok = mbar_wait(smem_u32(&bars->st_full[sn]), ((st_it + 1) / Cfg::kStages) & 1, abort,
                           a.status);
            if (!ok) break;
            tc_fence_after();
            issue_kq(tmem + kColS, sK, next);  // S^T(u+1)
            mma_commit(smem_u32(&bars->s_full));
          }
          ok = mbar_wait(smem_u32(&bars->ds_ready), it & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
          if constexpr (!DQ) {  // no dQ product: dK reads dS^T from TMEM
            issue_acc(tmem + Cfg::col_dk(), tmem + kColDP, stage, u > 0);  // dK += dS^T Q
          } else if constexpr (CAUSAL) {  // measured faster causal: dK first, dS^T from TMEM
            issue_acc(tmem + Cfg::col_dk(), tmem + kColDP, stage, u > 0);  // dK += dS^T Q
            issue_dq();                                                    // dQ_i = dS K
            mma_commit(smem_u32(&bars->dq_full));
          } else {
            issue_dq();  // dQ_i = dS K, read out while dK runs
            mma_commit(smem_u32(&bars->dq_full));
            issue_dk(stage, u > 0);  // dK += dS^T Q
          }
          mma_commit(smem_u32(&bars->st_empty[s]));
          if (!has_next) {
            mma_commit(smem_u32(&bars->acc_done));
            mma_commit(smem_u32(&bars->kv_empty));
          } else {
            if constexpr (DQ) {
              ok = mbar_wait(smem_u32(&bars->dq_free), it & 1, abort, a.status);
              if (!ok) break;
              tc_fence_after();
            }
            issue_kq(tmem + kColDP, sV, next + Cfg::kTileBytes);  // dP^T(u+1)
            mma_commit(smem_u32(&bars->dp_full));
          }
        }
      }
      mma_commit(smem_u32(&bars->drain));
      mbar_drain(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  }
  } else if (warp < kBwdDqWarp0) {
    // -------------------------------- compute warps: P^T and dS^T, 64 queries each
    const int wg = warp >> 2;            // query columns 64 wg .. 64 wg + 63
    const int r = (warp & 3) * 32 + lane;  // key row within the block = TMEM lane
    const uint32_t t_lane = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16);
    const uint32_t tS = t_lane + kColS + 64 * wg;
    const uint32_t tDP = t_lane + kColDP + 64 * wg;
    const float sl2 = a.scale_log2;
    uint32_t st_it = 0, it = 0, kv_round = 0;
    bool ok = true;
    // row r of query block wg of dS^T in shared memory: 128-byte rows, 16-byte
    // chunks stored at chunk ^ (r & 7)
    const uint32_t ds_row = sDS + wg * kBlk + r * 128;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd, ++kv_round) {
      const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
      if (item >= n_eff) break;  // only in the last, partial round
      int bh, j;
      if constexpr (VAR) {
        if (a.sched != nullptr) {
          int b, h;
          sched_decode(sched_arrays(a.sched, a.n_seq, a.sched_P), a.n_seq, a.sched_P, a.g.H,
                       CAUSAL, false, item, b, h, j);
          bh = b * a.g.H + h;
        } else {
          decode_kv_item(item, a, CAUSAL, bh, j);
        }
      } else {
        decode_kv_item(item, a, CAUSAL, bh, j);
      }
      int n_it;
      KvWork w;
      int key_thr = 0;  // VAR: key row of this thread minus (nk - nq); >= 2^29 past nk
      if constexpr (VAR) {
        const Seq sq = seq_of(bh, a.g);
        w = var_kv_work(j, sq, CAUSAL);
        n_it = w.n_it;
        const int key = j * kTile + r;
        if (n_it == 0) {
          if (sq.nq == 0 && key < sq.nk) {  // keys of a sequence without queries: dK = dV = 0
            __nv_bfloat16* out = (wg == 0 ? a.dv : a.dk) +
                                 sq.bb * (wg == 0 ? a.sdv.batch : a.sdk.batch) +
                                 sq.hh * (wg == 0 ? a.sdv.head : a.sdk.head) +
                                 static_cast<int64_t>(sq.k0 + key) * (wg == 0 ? a.sdv.row : a.sdk.row);
            for (int c = 0; c < D; c += 8)
              *reinterpret_cast<uint4*>(out + c) = make_uint4(0u, 0u, 0u, 0u);
          }
          --kv_round;  // no K/V round for this item
          continue;
        }
        key_thr = key >= sq.nk ? (1 << 29) : (CAUSAL ? key - (sq.nk - sq.nq) : -(1 << 29));
      } else {
        n_it = n_q - (CAUSAL ? j : 0);
      }
      for (int u = 0; u < n_it; ++u, ++it, ++st_it) {
        int i;
        if constexpr (VAR)
          i = var_qblock(w, u, CAUSAL);
        else
          i = qblock_at(j, u, n_q, CAUSAL);
        const uint32_t s = st_it % Cfg::kStages;
        const float* lse2 = reinterpret_cast<const float*>(smem + Cfg::kOffStages +
                                                           s * Cfg::kStageBytes +
                                                           2 * Cfg::kTileBytes) + 64 * wg;
        const float* Dq = lse2 + 128;
        // phase A: P^T = exp2(S^T * scale*log2e - lse2[q]), causal mask on the diagonal
        ok = mbar_wait_warp(smem_u32(&bars->s_full), it & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64(tS, sr);
        const int qlo = 64 * wg;
        // query columns below thr are masked for this key row
        int thr = r;
        bool diag = CAUSAL && i == j;
        if constexpr (VAR) {
          thr = key_thr - i * kTile;
          diag = thr > qlo;
        }
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 l2 = *reinterpret_cast<const float2*>(lse2 + 2 * c);
          const float2 x = ffma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])),
                                 make_float2(sl2, sl2), make_float2(-l2.x, -l2.y));
          float p0 = ex2_approx(x.x);
          float p1 = ex2_approx(x.y);
          if (diag) {  // query q sees key r only if r <= q (+ nk - nq)
            p0 = (qlo + 2 * c < thr) ? 0.f : p0;
            p1 = (qlo + 2 * c + 1 < thr) ? 0.f : p1;
          }
          pk[c] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tS, pk);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_ready));
        // phase B: dS^T = P^T o (dP^T - D[q]); the previous dQ MMA is done with
        // the dS buffer (its completion precedes dP^T(i) in MMA order)
        ok = mbar_wait_warp(smem_u32(&bars->dp_full), it & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        // two chunks of 32 queries: dP^T in, dS^T out to TMEM and shared memory
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dp[32];
          tmem_ld32(tDP + 32 * h, dp);
          uint32_t ds[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 pf =
                __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[16 * h + c]));
            const float2 dd = *reinterpret_cast<const float2*>(Dq + 32 * h + 2 * c);
            const float2 g = fadd2(make_float2(__uint_as_float(dp[2 * c]), __uint_as_float(dp[2 * c + 1])),
                                   make_float2(-dd.x, -dd.y));
            const float2 v = fmul2(pf, g);
            ds[c] = pack_bf16x2(v.x, v.y);
          }
          // the causal dK (and without dQ every dK) reads dS^T from TMEM
          if constexpr (CAUSAL || !DQ) tmem_st16(tDP + 16 * h, ds);
          if constexpr (DQ) {
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
              const int ch = 4 * h + u4;
              const uint32_t addr = ds_row + ((ch ^ (r & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(ds[4 * u4]),
                           "r"(ds[4 * u4 + 1]), "r"(ds[4 * u4 + 2]), "r"(ds[4 * u4 + 3])
                           : "memory");
            }
          }
        }
        if constexpr (DQ) fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->ds_ready));
      }
      if (!ok) break;
      // epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK
      ok = mbar_wait_warp(smem_u32(&bars->acc_done), kv_round & 1, abort, a.status);
      if (!ok) break;
      tc_fence_after();
      const int key = j * kTile + r;
      bool store;
      __nv_bfloat16* out;
      if constexpr (VAR) {
        const Seq sq = seq_of(bh, a.g);
        store = key < sq.nk;
        const Strides& so = wg == 0 ? a.sdv : a.sdk;
        out = (wg == 0 ? a.dv : a.dk) + sq.bb * so.batch + sq.hh * so.head +
              static_cast<int64_t>(sq.k0 + key) * so.row;
#ifdef FA_DEBUG
        if (store)
          store = fa_dcheck(in_span(so, a.g.cu_q != nullptr ? 1 : a.BH / a.g.H, a.g.H, a.g.rows_k,
                                    D, out - (wg == 0 ? a.dv : a.dk), D) &&
                                FA_IN_RANGE(sq.k0 + key, a.g.rows_k),
                            a.status);
#endif
      } else {
        store = key < a.N;
        out = wg == 0 ? a.dv + row_offset(a.sdv, bh, a.H, key)
                      : a.dk + row_offset(a.sdk, bh, a.H, key);
#ifdef FA_DEBUG
        if (store)
          store = fa_dcheck(in_span(wg == 0 ? a.sdv : a.sdk, a.BH / a.H, a.H, a.N, D,
                                    out - (wg == 0 ? a.dv : a.dk), D),
                            a.status);
#endif
      }
      const float mul = wg == 0 ? 1.f : a.scale;
      const uint32_t col = wg == 0 ? kColDV : Cfg::col_dk();
      if constexpr (VAR && D <= 64) {
        // Packed batches at d <= 64, whose items are short: staged through
        // the dS^T buffer, free once acc_done has fired (the last MMAs that
        // read it are complete). Each warp puts its 32 rows of a 64-column
        // block there and stores them back with whole row segments per
        // instruction. Measured on GB300, the packed d = 64 batch's backward
        // got 4.4% faster non-causal and 1.1% causal. Elsewhere it was not
        // faster (the packed d = 128 batch 2.2% slower non-causal, the dense
        // d = 128 kernel 0.6%): there the epilogue waits mostly behind the
        // last query block's dQ reductions, which pass through the same path
        // from the SM to L2.
        const uint32_t stg = sDS + wg * kBlk + (warp & 3) * 32 * 128;  // 32 rows x 128 B
        // the warp's rows are consecutive keys: row rr is (rr - lane) rows from this one
        const int64_t rstride = wg == 0 ? a.sdv.row : a.sdk.row;
#pragma unroll
        for (int cb = 0; cb < (D + 63) / 64; ++cb) {
          constexpr int kFull = D / 64;
          const int ncols = cb < kFull ? 64 : D - 64 * kFull;  // 64, or 32 at d = 32 and 96
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (32 * h >= ncols) break;
            uint32_t v[32];
            tmem_ld32(t_lane + col + 64 * cb + 32 * h, v);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int c = 4 * h + q;
              const uint32_t addr = stg + lane * 128 + ((c ^ (lane & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                           "r"(pack_bf16x2(__uint_as_float(v[8 * q + 0]) * mul,
                                           __uint_as_float(v[8 * q + 1]) * mul)),
                           "r"(pack_bf16x2(__uint_as_float(v[8 * q + 2]) * mul,
                                           __uint_as_float(v[8 * q + 3]) * mul)),
                           "r"(pack_bf16x2(__uint_as_float(v[8 * q + 4]) * mul,
                                           __uint_as_float(v[8 * q + 5]) * mul)),
                           "r"(pack_bf16x2(__uint_as_float(v[8 * q + 6]) * mul,
                                           __uint_as_float(v[8 * q + 7]) * mul))
                           : "memory");
            }
          }
          __syncwarp();
          // ncols / 8 lanes per row, 32 / (ncols / 8) rows per instruction
          const int cpr = ncols / 8, rpi = 32 / cpr;
#pragma unroll 1
          for (int k = 0; k < cpr; ++k) {
            const int rr = k * rpi + lane / cpr, c = lane % cpr;
            uint4 val;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                         : "r"(stg + rr * 128 + ((c ^ (rr & 7)) << 4))
                         : "memory");
            const int ok_row = __shfl_sync(0xffffffffu, static_cast<int>(store), rr);
            if (ok_row)
              *reinterpret_cast<uint4*>(out + (rr - lane) * rstride + 64 * cb + 8 * c) = val;
          }
          __syncwarp();
        }
      } else {
        // one row per thread, 64-byte pieces
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(t_lane + col + cc * 32, v);
          if (store) {
            uint4* dst = reinterpret_cast<uint4*>(out + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(v[8 * v4 + 0]) * mul, __uint_as_float(v[8 * v4 + 1]) * mul);
              w.y = pack_bf16x2(__uint_as_float(v[8 * v4 + 2]) * mul, __uint_as_float(v[8 * v4 + 3]) * mul);
              w.z = pack_bf16x2(__uint_as_float(v[8 * v4 + 4]) * mul, __uint_as_float(v[8 * v4 + 5]) * mul);
              w.w = pack_bf16x2(__uint_as_float(v[8 * v4 + 6]) * mul, __uint_as_float(v[8 * v4 + 7]) * mul);
              dst[v4] = w;
            }
          }
        }
      }
      // the next item's first dV/dK MMAs overwrite these accumulators only
      // after p_ready/ds_ready of that item, which these warps signal later
    }
  } else {
    // ------------------------------------------------- dQ warps: add dQ_i
    setmaxnreg_inc<176>();
    if constexpr (DQ) {
      const int wq = warp & 3;
      const uint32_t t_lane = tmem + ((static_cast<uint32_t>(wq) * 32u) << 16);
      uint32_t it = 0;
      bool ok = true;
      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= n_eff) break;  // only in the last, partial round
        int bh, j;
        if constexpr (VAR) {
          if (a.sched != nullptr) {
            int b, h;
            sched_decode(sched_arrays(a.sched, a.n_seq, a.sched_P), a.n_seq, a.sched_P, a.g.H,
                         CAUSAL, false, item, b, h, j);
            bh = b * a.g.H + h;
          } else {
            decode_kv_item(item, a, CAUSAL, bh, j);
          }
        } else {
          decode_kv_item(item, a, CAUSAL, bh, j);
        }
        int n_it, nq_rows;
        KvWork w;
        float* acc_base;  // accumulator row 0 of this (sequence, head)
        if constexpr (VAR) {
          const Seq sq = seq_of(bh, a.g);
          w = var_kv_work(j, sq, CAUSAL);
          n_it = w.n_it;
          nq_rows = sq.nq;
          acc_base = a.ws + 2 * static_cast<size_t>(a.planes) * a.lpad +
                     ((static_cast<size_t>(sq.bb) * a.g.H + sq.hh) * a.g.rows_q + sq.q0) * D;
        } else {
          n_it = CAUSAL ? n_q - j : n_q;
          nq_rows = a.N;
          acc_base = a.ws.dq_acc(a.BH, a.Npad) + static_cast<size_t>(bh) * a.N * D;
        }
        for (int u = 0; u < n_it; ++u, ++it) {
          int i;
          if constexpr (VAR)
            i = var_qblock(w, u, CAUSAL);
          else
            i = qblock_at(j, u, n_q, CAUSAL);
          ok = mbar_wait_warp(smem_u32(&bars->dq_full), it & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
          if constexpr (Cfg::kDqTransposed) {
            // lane = head-dim index dd, columns = the 128 queries of block i.
            // All 128 columns go to registers first and TMEM is released
            // before any atomic is issued, so the next dP^T never waits on them.
            int rows = min(kTile, nq_rows - i * kTile);
            if (!fa_dcheck(rows <= 0 || FA_IN_RANGE(i * kTile + rows - 1, nq_rows), a.status))
              rows = 0;  // debug build: the rows added lie inside the sequence's accumulator
            if constexpr (Cfg::kDupK) {
              // d = 64: warps 0 and 2 hold head dims 0-31, warps 1 and 3 dims
              // 32-63 (rows 64-127 repeat rows 0-63); warps 0, 1 add query
              // columns 0-63, warps 2, 3 columns 64-127
              const int dd = (wq & 1) * 32 + lane;
              const int qh = (wq >> 1) * 64;
              float* dst = acc_base + (static_cast<size_t>(i) * kTile + qh) * D + dd;
              uint32_t v[64];
              tmem_ld64(t_lane + kColDP + qh, v);
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
#pragma unroll
              for (int q = 0; q < 64; ++q)
                if (qh + q < rows) atomicAdd(dst + static_cast<size_t>(q) * D, __uint_as_float(v[q]));
              continue;
            }
            const int dd = wq * 32 + lane;
            float* dst = acc_base + static_cast<size_t>(i) * kTile * D + dd;
            uint32_t v[64], w[64];
            tmem_ld64(t_lane + kColDP, v);
            tmem_ld64(t_lane + kColDP + 64, w);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
            if (wq * 32 < D) {  // whole warps of head-dim rows past d hold zeros
#pragma unroll
              for (int q = 0; q < 64; ++q)
                if (q < rows) atomicAdd(dst + static_cast<size_t>(q) * D, __uint_as_float(v[q]));
#pragma unroll
              for (int q = 0; q < 64; ++q)
                if (64 + q < rows)
                  atomicAdd(dst + static_cast<size_t>(64 + q) * D, __uint_as_float(w[q]));
            }
          } else {
            // lane = query row, columns = the d head-dim values
            uint32_t v[D];
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t t32[32];
              tmem_ld32(t_lane + kColDP + c0, t32);
#pragma unroll
              for (int u = 0; u < 32; ++u) v[c0 + u] = t32[u];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
            const int row = i * kTile + wq * 32 + lane;
            if (row < nq_rows) {
              float4* dst = reinterpret_cast<float4*>(acc_base + static_cast<size_t>(row) * D);
#pragma unroll
              for (int c = 0; c < D / 4; ++c)
                atomicAdd(dst + c, make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                               __uint_as_float(v[4 * c + 2]),
                                               __uint_as_float(v[4 * c + 3])));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kBwdMmaWarp) tmem_dealloc(tmem, kBwdTmemCols);
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_t(const Problem& p, const CUtensorMap* maps, const PreArgs& pa,
                         const BwdArgs& a, const DqArgs& qa, int stages, cudaStream_t stream) {
  if (stages & kStagePre) {
    const size_t work = static_cast<size_t>(a.BH) * a.Npad * (D <= 32 ? 4 : (D <= 64 ? 8 : (D <= 128 ? 16 : 32)));
    const int grid = static_cast<int>(std::min<size_t>((work + 255) / 256, static_cast<size_t>(p.num_sms) * 8));
    bwd_pre_kernel<D><<<grid, 256, 0, stream>>>(pa);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kStageDkdv) {
    if constexpr (D == 256) {  // its own kernel over 64-key blocks (fa_bwd256.cu)
      Bwd256Args b;
      b.lse2 = a.ws.lse2(a.BH, a.Npad);
      b.Drow = a.ws.Drow(a.BH, a.Npad);
      b.dq_acc = a.ws.dq_acc(a.BH, a.Npad);
      b.dk = a.dk;
      b.dv = a.dv;
      b.status = a.status;
      b.N = a.N;
      b.H = a.H;
      b.Npad = a.Npad;
      b.BH = a.BH;
      b.n_kb = (a.N + 63) / 64;
      b.n_qb = a.n_tiles;
      b.n_items = a.BH * b.n_kb;
      b.scale = a.scale;
      b.scale_log2 = a.scale_log2;
      b.sdk = a.sdk;
      b.sdv = a.sdv;
      const cudaError_t e = launch_bwd256_dkdv(p, maps[0], maps[1], maps[2], maps[3], b, stream);
      if (e != cudaSuccess) return e;
    } else {
      constexpr int smem = bwd_smem_bytes<D>();
      auto kern = bwd_dkdv_kernel<D, CAUSAL, false, true>;
      if constexpr (D == 64 || D == 128) {
        if (p.dq_separate) kern = bwd_dkdv_kernel<D, CAUSAL, false, false>;
      }
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      const int grid = min(a.n_items, p.num_sms);
      kern<<<grid, kBwdThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], a);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  if ((stages & kStageDq) && p.dq_separate) {  // the query-stationary dQ kernel (fa_bwd_dq.cu)
    BwdDqArgs b;
    b.lse2 = a.ws.lse2(a.BH, a.Npad);
    b.Drow = a.ws.Drow(a.BH, a.Npad);
    b.dq = qa.dq;
    b.status = a.status;
    b.N = a.N;
    b.H = a.H;
    b.Npad = a.Npad;
    b.BH = a.BH;
    b.n_tiles = a.n_tiles;
    b.n_items = a.BH * a.n_tiles;
    b.scale = a.scale;
    b.scale_log2 = a.scale_log2;
    b.sdq = qa.sdq;
    return launch_bwd_dq_separate(p, maps, b, stream);
  }
  if (stages & kStageDq) {
    const size_t n8 = static_cast<size_t>(a.BH) * a.N * D / 8;
    const int grid = static_cast<int>(std::min<size_t>((n8 + 255) / 256, static_cast<size_t>(p.num_sms) * 8));
    dq_convert_kernel<D><<<grid, 256, 0, stream>>>(qa, n8);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_var_t(const Problem& p, const CUtensorMap* maps, const PreVarArgs& pa,
                             const BwdVarArgs& a, const DqArgs& qa, cudaStream_t stream) {
  {
    const size_t work = static_cast<size_t>(pa.BH) * pa.max_q_pad * (D <= 32 ? 4 : (D <= 64 ? 8 : (D <= 128 ? 16 : 32)));
    const int grid = static_cast<int>(std::min<size_t>((work + 255) / 256, static_cast<size_t>(p.num_sms) * 8));
    bwd_pre_var_kernel<D><<<grid, 256, 0, stream>>>(pa);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.sched != nullptr) {
    bwd_var_sched_kernel<CAUSAL><<<1, kSchedBuildThreads, 0, stream>>>(a.g, a.n_seq, a.sched_P,
                                                                       a.sched);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    constexpr int smem = bwd_smem_bytes<D>();
    auto kern = bwd_dkdv_kernel<D, CAUSAL, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int grid = min(a.n_items, p.num_sms);
    kern<<<grid, kBwdThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const size_t n8 = static_cast<size_t>(qa.BH) * qa.N * D / 8;
  const int grid = static_cast<int>(std::min<size_t>((n8 + 255) / 256, static_cast<size_t>(p.num_sms) * 8));
  dq_convert_kernel<D><<<grid, 256, 0, stream>>>(qa, n8);
  return cudaGetLastError();
}

cudaError_t launch_bwd_var(const Problem& p, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dO, void* dq, void* dk,
                           void* dv, void* workspace, cudaStream_t stream) {
  const bool packed = p.cu_q != nullptr;
  const int planes_b = packed ? 1 : p.B;
  CUtensorMap maps[4];
  if (!make_tile_map(&maps[0], q, planes_b, p.H, p.rows_q, p.d, p.st[kQ]) ||
      !make_tile_map(&maps[1], k, planes_b, p.H, p.rows_k, p.d, p.st[kK]) ||
      !make_tile_map(&maps[2], v, planes_b, p.H, p.rows_k, p.d, p.st[kV]) ||
      !make_tile_map(&maps[3], dO, planes_b, p.H, p.rows_q, p.d, p.st[kdO]))
    return cudaErrorInvalidValue;
  const VarGeom g{p.cu_q, p.cu_k, p.H, p.N, p.Nk, p.rows_q, p.rows_k, p.max_q, p.max_k};
  const int planes = planes_b * p.H;
  const int lpad = var_padded_rows(packed, p.B, p.rows_q);
  float* ws = static_cast<float*>(workspace);
  PreVarArgs pa;
  pa.o = static_cast<const __nv_bfloat16*>(o);
  pa.dO = static_cast<const __nv_bfloat16*>(dO);
  pa.lse = lse;
  pa.ws = ws;
  pa.so = p.st[kO];
  pa.sdo = p.st[kdO];
  pa.planes = planes;
  pa.lpad = lpad;
  pa.max_q_pad = (p.max_q + kTile - 1) / kTile * kTile;
  pa.BH = p.B * p.H;
  pa.g = g;
  BwdVarArgs a;
  a.ws = ws;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.status = p.status;
  a.BH = p.B * p.H;
  a.n_tiles = (p.max_k + kTile - 1) / kTile;
  a.n_items = a.BH * a.n_tiles;
  a.planes = planes;
  a.lpad = lpad;
  a.scale = p.scale;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.sdk = p.st[kdK];
  a.sdv = p.st[kdV];
  a.g = g;
  a.n_seq = p.B;
  a.sched_P = (p.max_k + kTile - 1) / kTile;
  // packed: the schedule's arrays after the accumulator (16-byte aligned)
  a.sched = packed ? reinterpret_cast<int*>(
                         ws + 2 * static_cast<size_t>(planes) * lpad +
                         (static_cast<size_t>(planes) * p.rows_q * p.d + 3) / 4 * 4)
                   : nullptr;
  DqArgs qa;  // the accumulator as planes x rows_q rows after 2 x planes x lpad floats
  qa.ws = Workspace{ws};
  qa.dq = static_cast<__nv_bfloat16*>(dq);
  qa.sdq = p.st[kdQ];
  qa.N = p.rows_q;
  qa.H = p.H;
  qa.Npad = lpad;
  qa.BH = planes;
  qa.scale = p.scale;
  qa.status = p.status;
  switch (p.d) {
    case 32:
      return p.causal ? launch_bwd_var_t<32, true>(p, maps, pa, a, qa, stream)
                      : launch_bwd_var_t<32, false>(p, maps, pa, a, qa, stream);
    case 64:
      return p.causal ? launch_bwd_var_t<64, true>(p, maps, pa, a, qa, stream)
                      : launch_bwd_var_t<64, false>(p, maps, pa, a, qa, stream);
    case 96:
      return p.causal ? launch_bwd_var_t<96, true>(p, maps, pa, a, qa, stream)
                      : launch_bwd_var_t<96, false>(p, maps, pa, a, qa, stream);
    default:
      return p.causal ? launch_bwd_var_t<128, true>(p, maps, pa, a, qa, stream)
                      : launch_bwd_var_t<128, false>(p, maps, pa, a, qa, stream);
  }
}

}  // namespace

size_t bwd_var_workspace_bytes(bool packed, int B, int H, int rows_q, int max_k, int d) {
  const size_t planes = static_cast<size_t>(packed ? 1 : B) * H;
  const size_t lpad = static_cast<size_t>(var_padded_rows(packed, B, rows_q));
  const size_t acc = (planes * static_cast<size_t>(rows_q) * d + 3) / 4 * 4;
  // packed: the compacted schedule's arrays after the accumulator, then the
  // builder's scratch
  const int P = (max_k + kTile - 1) / kTile;
  const size_t sched = packed ? sched_ints(B, P) + sched_build_scratch_ints(P) : 0;
  return (2 * planes * lpad + acc + sched) * 4;
}

size_t bwd_workspace_bytes(int B, int H, int N, int d) {
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t Npad = (static_cast<size_t>(N) + kTile - 1) / kTile * kTile;
  return 2 * BH * Npad * 4 + BH * static_cast<size_t>(N) * d * 4;
}

cudaError_t launch_bwd(const Problem& p, const void* q, const void* k, const void* v,
                       const void* o, const float* lse, const void* dO, void* dq, void* dk,
                       void* dv, void* workspace, int stages, cudaStream_t stream) {
  if (p.var) {
    if (stages != kStagesAll) return cudaErrorInvalidValue;
    return launch_bwd_var(p, q, k, v, o, lse, dO, dq, dk, dv, workspace, stream);
  }
  const int BH = p.B * p.H;
  CUtensorMap maps[4];
  const int kv_rows = p.d == 256 ? 64 : kTile;  // the d = 256 kernel takes 64-key blocks
  // and loads whole tiles with 5-D copies (q causal: in two halves)
  const int blocks = p.d == 256 ? 4 : 1;
  if (p.dq_separate && !bwd_dq_separate_supported(p.d)) return cudaErrorInvalidValue;
  if ((stages & (p.dq_separate ? (kStageDkdv | kStageDq) : kStageDkdv)) &&
      (!make_tile_map(&maps[0], q, p.B, p.H, p.N, p.d, p.st[kQ], kTile,
                      p.d == 256 && p.causal ? 2 : blocks) ||
       !make_tile_map(&maps[1], k, p.B, p.H, p.N, p.d, p.st[kK], kv_rows, blocks) ||
       !make_tile_map(&maps[2], v, p.B, p.H, p.N, p.d, p.st[kV], kv_rows, blocks) ||
       !make_tile_map(&maps[3], dO, p.B, p.H, p.N, p.d, p.st[kdO], kTile, blocks)))
    return cudaErrorInvalidValue;
  const int n_tiles = (p.N + kTile - 1) / kTile;
  const Workspace ws{static_cast<float*>(workspace)};
  PreArgs pa;
  pa.o = static_cast<const __nv_bfloat16*>(o);
  pa.dO = static_cast<const __nv_bfloat16*>(dO);
  pa.lse = lse;
  pa.ws = ws;
  pa.so = p.st[kO];
  pa.sdo = p.st[kdO];
  pa.N = p.N;
  pa.H = p.H;
  pa.Npad = n_tiles * kTile;
  pa.BH = BH;
  pa.zero_acc = p.dq_separate ? 0 : 1;
  BwdArgs a;
  a.ws = ws;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.status = p.status;
  a.N = p.N;
  a.H = p.H;
  a.Npad = n_tiles * kTile;
  a.BH = BH;
  a.n_tiles = n_tiles;
  a.n_items = BH * n_tiles;
  a.scale = p.scale;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.sdk = p.st[kdK];
  a.sdv = p.st[kdV];
  DqArgs qa;
  qa.ws = ws;
  qa.dq = static_cast<__nv_bfloat16*>(dq);
  qa.sdq = p.st[kdQ];
  qa.N = p.N;
  qa.H = p.H;
  qa.Npad = n_tiles * kTile;
  qa.BH = BH;
  qa.scale = p.scale;
  qa.status = p.status;
  switch (p.d) {
    case 32:
      return p.causal ? launch_bwd_t<32, true>(p, maps, pa, a, qa, stages, stream)
                      : launch_bwd_t<32, false>(p, maps, pa, a, qa, stages, stream);
    case 64:
      return p.causal ? launch_bwd_t<64, true>(p, maps, pa, a, qa, stages, stream)
                      : launch_bwd_t<64, false>(p, maps, pa, a, qa, stages, stream);
    case 96:
      return p.causal ? launch_bwd_t<96, true>(p, maps, pa, a, qa, stages, stream)
                      : launch_bwd_t<96, false>(p, maps, pa, a, qa, stages, stream);
    case 256:
      return p.causal ? launch_bwd_t<256, true>(p, maps, pa, a, qa, stages, stream)
                      : launch_bwd_t<256, false>(p, maps, pa, a, qa, stages, stream);
    default:
      return p.causal ? launch_bwd_t<128, true>(p, maps, pa, a, qa, stages, stream)
                      : launch_bwd_t<128, false>(p, maps, pa, a, qa, stages, stream);
  }
}

}  // namespace fa

// Forward kernel: exact attention, tile by tile, with an online softmax.
//
// What it computes ("flashattention-2" glossary, "How FlashAttention-2 Works
// (Tiled Algorithm)"; "Flash Attention v2" notes, "Detailed Algorithm
// Comparison", forward pass): for each 128-row query tile Q_i, stream the
// 128-key tiles K_j, V_j; S = Q_i K_j^T; keep a running row max m and row sum
// l; P = exp(scale*S - scale*m); O = alpha*O + P V_j with alpha =
// exp(scale*(m_old - m_new)); at the end O / l and lse = scale*m + ln l.
//
// GB300 mapping (not the pages' A100 scheme):
//  - persistent CTAs, one per SM, each taking work items (batch*head, pair
//    of query tiles) in a static stride; causal items longest first
//    ("FlashAttention-2 paper" digest, "Three changes": query blocks of one
//    head are split across thread blocks; glossary improvements table,
//    "Causal Masking": fully masked tiles skipped);
//  - warp 8 issues TMA loads of Q (once per item) and of K/V tiles into a
//    ring of shared-memory stages guarded by full/empty mbarriers;
//  - warp 9 issues tcgen05.mma: S_t = Q_t K_j^T into tensor memory (TMEM),
//    then O_t += P_t V_j with P_t read from TMEM (P overwrites S in place);
//  - warps 0-3 and 4-7 are two softmax warpgroups, one per query tile, one
//    thread per query row (the TMEM lane of that row). While one warpgroup
//    runs its softmax the tensor core works on the other tile's products;
//  - the rescale of O is deferred: it is applied only when the row maximum
//    grows by more than kRescaleTauLog2 (in log2 units; 0 = every growth).
//    O and l are always scaled by the same factor, so the result is exact in
//    real arithmetic ("FlashAttention-2 paper" digest, "Three changes": the
//    rescaling is delayed and batched). 1/l is applied once in the epilogue.
//
// TMEM (512 columns x 128 lanes of 32 bit): S0 [0,128), S1 [128,256),
// O0 [256, 256+d), O1 [256+d, 256+2d). P_t is bf16, two per column, in the
// first 64 columns of S_t.

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "schedule.cuh"
#include "seq.cuh"

namespace fa {
namespace {

#ifndef FA_RESCALE_TAU_LOG2
#define FA_RESCALE_TAU_LOG2 8.0f
#endif
constexpr float kRescaleTauLog2 = FA_RESCALE_TAU_LOG2;

// Of every 8 pairs of exponentials in a row, this many are evaluated by the
// FMA-pipe polynomial (exp2_poly2) instead of the MUFU ex2 unit. Measured on
// GB300 at d = 128, N = 4096: 0 -> 1107 TFLOP/s, 2 -> 1116, 3 -> 1089,
// 4 -> 1021, and 0 is best for causal and d = 64: the MUFU unit is not what
// bounds the softmax here, so the default keeps every exponential on it.
#ifndef FA_POLY_EXP_PAIRS_PER_8
#define FA_POLY_EXP_PAIRS_PER_8 0
#endif
constexpr int kPolyExpPairsPer8 = FA_POLY_EXP_PAIRS_PER_8;

constexpr int kFwdThreads = 320;  // 8 softmax warps + load warp + MMA warp
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr int kBlockBytes = kTile * 64 * 2;  // one 128-row x 64-column bf16 block: 16 KiB

template <int D>
struct FwdCfg {
  // head dims that are not a multiple of 64 (32, 96) use whole 64-column
  // blocks in shared memory; TMA zero-fills the columns past d and the MMAs
  // only read the first d
  static constexpr int kColBlocks = (D + 63) / 64;
  static constexpr int kTileBytes = kTile * kColBlocks * 64 * 2;
  static constexpr int kStages = (kColBlocks == 2) ? 4 : 8;
  static constexpr int kQBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kTileBytes;
  // TMEM column of S_t and of O_t
  __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __device__ static constexpr uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(D) * t; }
  // d <= 64 can keep Q_t in TMEM too (d / 2 columns of bf16 pairs, after O0
  // and O1), so that S_t = Q_t K^T reads only K from shared memory. The
  // tensor core's time is its shared-memory operand reads plus its math
  // (ncu: tensor pipe active + TC shared-memory wavefronts ~ 95-100% of the
  // elapsed time in every kernel here), so an A operand from TMEM shortens
  // each S product. At d = 96 and 128 the four S and O buffers fill TMEM.
  // Measured on GB300 against Q read from shared memory: non-causal 2.6%
  // faster at d = 64, N = 4096 (4.0% at N = 16384) and 1.9% at d = 32; the
  // causal and packed-batch instantiations ran 1.6% and 4% slower (the copy
  // adds registers where they were at the limit), so only the non-causal,
  // non-packed ones take it (fwd_kernel's kQT).
  static constexpr bool kQTmemFits = D <= 64;
  __device__ static constexpr uint32_t col_q(int t) {
    return 256u + 2u * static_cast<uint32_t>(D) + static_cast<uint32_t>(D / 2) * t;
  }
};
static_assert(FwdCfg<64>::col_q(1) + 32 <= 512 && FwdCfg<32>::col_q(1) + 16 <= 512,
              "Q in TMEM past the allocation");

struct FwdBarriers {
  uint64_t q_full[2], q_empty[2], q_tmem[2];
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
constexpr int fwd_smem_bytes() {
  return 1024 + FwdCfg<D>::kQBytes + FwdCfg<D>::kRingBytes + static_cast<int>(sizeof(FwdBarriers));
}

struct FwdArgs {
  __nv_bfloat16* o;
  float* lse;
  int* status;
  int N, H, BH, n_tiles, n_pairs, n_items;
  float scale, scale_log2;
  Strides so;  // element strides of o
};

// Arguments of the kernel for sequences of unequal lengths (dense or packed
// batch); sh = b * H + h runs over sequences and heads.
struct FwdVarArgs {
  __nv_bfloat16* o;
  float* lse;  // [planes, rows_q] with planes = batch coordinates x H
  int* status;
  int BH, n_pairs, n_items;  // BH = sequences x heads; pairs of the longest sequence
  int n_seq;    // sequences
  int compact;  // packed batch: compacted schedule built in shared memory
  float scale, scale_log2;
  Strides so;
  VarGeom g;
};

// Packed batches get the compacted, longest-first schedule (seq.cuh,
// Sched) when its arrays fit in the spare shared memory; the levels are the
// query-tile pairs, causal visited from the highest (the most key tiles).

template <bool VAR>
struct FwdArgsOf {
  using type = FwdArgs;
};
template <>
struct FwdArgsOf<true> {
  using type = FwdVarArgs;
};

// Decode with the keys split over work items (SPLIT, with VAR: a dense batch
// of Nq <= 16 query rows per sequence against a key/value cache, with or
// without per-sequence key counts). Item = (b*h, split s); split s covers an
// even share of the key tiles the sequence's rows see (split_tiles), and
// writes its rows' O normalised by its own row sum
// (fp32) and its log-sum-exp in log2 units into the decode workspace, which
// the decode combine kernel merges by log-sum-exp (the identity the online
// softmax rests on: "Flash Attention v2" notes, "Detailed Algorithm
// Comparison", forward pass). A split with no key tile writes -inf and 0.
struct FwdSplitArgs : FwdVarArgs {
  float* part_o;    // [B*H, splits, nq_pad, D]
  float* part_lse;  // [B*H, splits, nq_pad]
  int splits, nq_pad;
};

template <bool VAR, bool SPLIT>
struct FwdArgsSel {
  using type = typename FwdArgsOf<VAR>::type;
};
template <>
struct FwdArgsSel<true, true> {
  using type = FwdSplitArgs;
};

// SPLIT: the split's first key tile t0 and its number of key tiles, out of
// the J tiles the sequence's rows see from tile 0, divided evenly over the
// splits (so that sequences shorter than the cache keep every split busy).
__device__ __forceinline__ int split_tiles(const FwdSplitArgs& a, int split, int J, int& t0) {
  const int tps = (J + a.splits - 1) / a.splits;
  t0 = split * tps;
  return max(0, min(J - t0, tps));
}

template <class Args>
__device__ __forceinline__ void decode_item(int item, const Args& a, bool causal, int& bh,
                                            int& pair) {
  if (causal) {  // longest first: the last query pairs of every head come first
    pair = a.n_pairs - 1 - item / a.BH;
    bh = item % a.BH;
  } else {  // the pairs of one head are adjacent, so concurrent CTAs share K/V in L2
    bh = item / a.n_pairs;
    pair = item % a.n_pairs;
  }
}

// Number of K/V tiles query tile qt visits (0 if the tile lies past N).
__device__ __forceinline__ int tile_steps(int qt, const FwdArgs& a, bool causal) {
  if (qt >= a.n_tiles) return 0;
  return causal ? min(qt + 1, a.n_tiles) : a.n_tiles;
}

// The same for a sequence of unequal lengths. A tile whose rows see no key
// at all (causal with nq > nk, or nk = 0) still runs one fully masked step,
// which leaves l = 0: its rows get O = 0 and LSE = -inf.
__device__ __forceinline__ int var_tile_steps(int qt, const Seq& s, bool causal) {
  if (qt * kTile >= s.nq) return 0;
  const int nkt = (s.nk + kTile - 1) / kTile;
  int n = nkt;
  if (causal) {
    const int last_key = min(qt * kTile + kTile - 1, s.nq - 1) + s.nk - s.nq;
    n = last_key < 0 ? 0 : min(nkt, last_key / kTile + 1);
  }
  return max(n, 1);
}

template <int D, bool CAUSAL, bool VAR, bool COMPACT = false, bool KLENS = false,
          bool SPLIT = false>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV,
               const typename FwdArgsSel<VAR, SPLIT>::type a) {
  static_assert(!SPLIT || (VAR && !COMPACT), "the key split is decode's");
  using Cfg = FwdCfg<D>;
  constexpr bool kQT = Cfg::kQTmemFits && !CAUSAL && !COMPACT;  // Q_t in TMEM (FwdCfg)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + Cfg::kQBytes;
  FwdBarriers* bars = reinterpret_cast<FwdBarriers*>(smem + Cfg::kQBytes + Cfg::kRingBytes);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->q_full[t]), 1);
      // kQT: the softmax warps release Q's buffer once they have copied it
      mbar_init(smem_u32(&bars->q_empty[t]), kQT ? 4 : 1);
      mbar_init(smem_u32(&bars->q_tmem[t]), 4);
      mbar_init(smem_u32(&bars->s_full[t]), 1);
      mbar_init(smem_u32(&bars->p_full[t]), 4);  // one elected lane per softmax warp
      mbar_init(smem_u32(&bars->o_done[t]), 1);
    }
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  Sched sched{};          // compacted schedule of a packed batch (VAR && COMPACT)
  int n_eff = a.n_items;  // items of the schedule
  if constexpr (VAR && COMPACT) {
    sched = sched_arrays(reinterpret_cast<int*>(smem + Cfg::kQBytes + Cfg::kRingBytes +
                                                ((sizeof(FwdBarriers) + 15) / 16) * 16),
                         a.n_seq, a.n_pairs);
    // scratch: the K/V ring, which no copy uses before the roles start
    build_sched(
        sched, a.n_seq, a.n_pairs, a.g.H, CAUSAL, /*top_first=*/true,
        [&](int b) { return (seq_of(b * a.g.H, a.g).nq + 2 * kTile - 1) / (2 * kTile); },
        reinterpret_cast<int*>(smem + Cfg::kQBytes), Cfg::kRingBytes / 4);
    n_eff = sched_total(sched, a.n_seq, a.n_pairs, CAUSAL);
    fence_proxy_async_smem();  // before TMA writes into the ring
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t kv_it = 0;
      uint32_t q_issued[2] = {0u, 0u};
      bool ok = true;
      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= n_eff) break;  // only in the last, partial round
        int bh, pair, split = 0;
        if constexpr (VAR && COMPACT) {
          int b, h;
          sched_decode(sched, a.n_seq, a.n_pairs, a.g.H, CAUSAL, true, item, b, h, pair);
          bh = b * a.g.H + h;
        } else if constexpr (SPLIT) {
          bh = item / a.splits;
          split = item - bh * a.splits;
          pair = 0;
        } else {
          decode_item(item, a, CAUSAL, bh, pair);
        }
        int hh, bb, q0 = 0, k0 = 0, J, t0 = 0;
        if constexpr (VAR) {
          const Seq sq = seq_of<KLENS>(bh, a.g);
          hh = sq.hh;
          bb = sq.bb;
          q0 = sq.q0;
          k0 = sq.k0;
          J = max(var_tile_steps(2 * pair, sq, CAUSAL), var_tile_steps(2 * pair + 1, sq, CAUSAL));
          if constexpr (SPLIT) J = split_tiles(a, split, J, t0);
          if (J == 0) continue;  // every tile of the pair lies past the sequence
        } else {
          hh = bh % a.H;
          bb = bh / a.H;
          J = max(tile_steps(2 * pair, a, CAUSAL), tile_steps(2 * pair + 1, a, CAUSAL));
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          ok = mbar_wait(smem_u32(&bars->q_empty[t]), (q_issued[t] & 1) ^ 1, abort, a.status);
          if (!ok) break;
          const uint32_t bar = smem_u32(&bars->q_full[t]);
          mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
          for (int cb = 0; cb < Cfg::kColBlocks; ++cb)
            tma_load_4d(sQ + (t * Cfg::kColBlocks + cb) * kBlockBytes, &tmQ, bar, 64 * cb,
                        q0 + (2 * pair + t) * kTile, hh, bb, pol_q);
          ++q_issued[t];
        }
        for (int j = 0; j < J && ok; ++j) {
          for (int w = 0; w < 2; ++w) {  // K_j then V_j
            const uint32_t s = kv_it % Cfg::kStages;
            ok = mbar_wait(smem_u32(&bars->kv_empty[s]), ((kv_it / Cfg::kStages) & 1) ^ 1, abort,
                           a.status);
            if (!ok) break;
            const uint32_t bar = smem_u32(&bars->kv_full[s]);
            mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
            for (int cb = 0; cb < Cfg::kColBlocks; ++cb)
              tma_load_4d(sKV + (s * Cfg::kColBlocks + cb) * kBlockBytes, w ? &tmV : &tmK, bar,
                          64 * cb, k0 + (t0 + j) * kTile, hh, bb, pol_kv);
            ++kv_it;
          }
        }
      }
      // Producer tail. Normal path: wait until the consumer has released every
      // stage, so that no barrier arrival lands after the CTA exits. After an
      // abort: wait (bounded) for the copies already issued to land.
      const uint32_t n = min(kv_it, static_cast<uint32_t>(Cfg::kStages));
      for (uint32_t i = kv_it - n; i < kv_it; ++i) {
        const uint32_t s = i % Cfg::kStages, ph = (i / Cfg::kStages) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->kv_empty[s]), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->kv_full[s]), ph, 100000000ull);
      }
      for (int t = 0; t < 2; ++t) {
        if (q_issued[t] == 0) continue;
        const uint32_t ph = (q_issued[t] - 1) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->q_empty[t]), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->q_full[t]), ph, 100000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kTile, D, false, true);
      uint32_t kv_it = 0, q_round = 0;
      uint32_t step[2] = {0u, 0u};
      uint32_t qt_round[2] = {0u, 0u};  // kQT: Q copies into TMEM waited for, per tile
      bool ok = true;

      // S_t = Q_t K^T over d in steps of 16
      // descriptors are built once per tile; a K step adds a constant
      const SmemDesc dq[2] = {make_desc_sw128(sQ, 16, 1024),
                              make_desc_sw128(sQ + Cfg::kTileBytes, 16, 1024)};
      auto issue_s = [&](int t, uint32_t slot) {
        const uint32_t dst = tmem + Cfg::col_s(t);
        const SmemDesc da = dq[t];
        const SmemDesc db = make_desc_sw128(sKV + slot * Cfg::kTileBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
          if constexpr (kQT)  // Q_t from TMEM: 8 columns per 16 head dims
            mma_ts(dst, tmem + Cfg::col_q(t) + 8 * kk, desc_at(db, off), idesc_s, kk > 0);
          else
            mma_ss(dst, desc_at(da, off), desc_at(db, off), idesc_s, kk > 0);
        }
      };
      // O_t (+)= P_t V over the 128 keys in steps of 16
      auto issue_pv = [&](int t, uint32_t slot, bool accumulate) {
        const uint32_t dst = tmem + Cfg::col_o(t);
        const uint32_t pa = tmem + Cfg::col_s(t);
        const SmemDesc db = make_desc_sw128(sKV + slot * Cfg::kTileBytes, kBlockBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(dst, pa + kk * 8, desc_at(db, kk * 2048), idesc_o,
                 (accumulate || kk > 0) ? 1u : 0u);
      };

      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd, ++q_round) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= n_eff) break;  // only in the last, partial round
        int bh, pair, split = 0;
        if constexpr (VAR && COMPACT) {
          int b, h;
          sched_decode(sched, a.n_seq, a.n_pairs, a.g.H, CAUSAL, true, item, b, h, pair);
          bh = b * a.g.H + h;
        } else if constexpr (SPLIT) {
          bh = item / a.splits;
          split = item - bh * a.splits;
          pair = 0;
        } else {
          decode_item(item, a, CAUSAL, bh, pair);
        }
        int Jt[2];
        if constexpr (VAR) {
          const Seq sq = seq_of<KLENS>(bh, a.g);
          Jt[0] = var_tile_steps(2 * pair, sq, CAUSAL);
          Jt[1] = var_tile_steps(2 * pair + 1, sq, CAUSAL);
          if constexpr (SPLIT) {
            int t0;
            Jt[0] = split_tiles(a, split, Jt[0], t0);
            Jt[1] = split_tiles(a, split, Jt[1], t0);
          }
          if (Jt[0] == 0 && Jt[1] == 0) {  // skipped by the loader too: no Q round
            --q_round;
            continue;
          }
        } else {
          Jt[0] = tile_steps(2 * pair, a, CAUSAL);
          Jt[1] = tile_steps(2 * pair + 1, a, CAUSAL);
        }
        const int J = max(Jt[0], Jt[1]);
        const uint32_t base = kv_it;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if constexpr (kQT) {  // the softmax warps copied Q_t into TMEM
            if (ok && Jt[t] > 0) {
              ok = mbar_wait(smem_u32(&bars->q_tmem[t]), qt_round[t] & 1, abort, a.status);
              ++qt_round[t];
            }
          } else {
            if (ok) ok = mbar_wait(smem_u32(&bars->q_full[t]), q_round & 1, abort, a.status);
          }
        }
        if (!ok) break;
        tc_fence_after();
        // K_0
        {
          const uint32_t s = base % Cfg::kStages;
          ok = mbar_wait(smem_u32(&bars->kv_full[s]), (base / Cfg::kStages) & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (Jt[t] > 0) {
              issue_s(t, s);
              mma_commit(smem_u32(&bars->s_full[t]));
            }
            if (!kQT && Jt[t] <= 1) mma_commit(smem_u32(&bars->q_empty[t]));
          }
          mma_commit(smem_u32(&bars->kv_empty[s]));
        }
        for (int j = 0; j < J && ok; ++j) {
          const uint32_t iv = base + 2 * j + 1, ik = base + 2 * j + 2;
          const uint32_t sv = iv % Cfg::kStages, sk = ik % Cfg::kStages;
          ok = mbar_wait(smem_u32(&bars->kv_full[sv]), (iv / Cfg::kStages) & 1, abort, a.status);
          if (!ok) break;
          bool k_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok || j >= Jt[t]) continue;
            ok = mbar_wait(smem_u32(&bars->p_full[t]), step[t] & 1, abort, a.status);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, sv, j > 0);
            mma_commit(smem_u32(&bars->o_done[t]));
            ++step[t];
            if (j + 1 < Jt[t]) {
              if (!k_ready) {
                ok = mbar_wait(smem_u32(&bars->kv_full[sk]), (ik / Cfg::kStages) & 1, abort,
                               a.status);
                if (!ok) break;
                tc_fence_after();
                k_ready = true;
              }
              issue_s(t, sk);
              mma_commit(smem_u32(&bars->s_full[t]));
              if (!kQT && j + 2 == Jt[t]) mma_commit(smem_u32(&bars->q_empty[t]));
            }
          }
          if (!ok) break;
          mma_commit(smem_u32(&bars->kv_empty[sv]));
          if (j + 1 < J) {
            if (!k_ready) {  // K_{j+1} loaded but used by no tile: release it anyway
              ok = mbar_wait(smem_u32(&bars->kv_full[sk]), (ik / Cfg::kStages) & 1, abort,
                             a.status);
              if (!ok) break;
            }
            mma_commit(smem_u32(&bars->kv_empty[sk]));
          }
        }
        kv_it = base + 2 * J;
      }
      // every MMA issued so far completes before TMEM is released
      mma_commit(smem_u32(&bars->drain));
      mbar_drain(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;            // query tile of this warpgroup
    const int r = (warp & 3) * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t t_lane = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16);
    const uint32_t tS = t_lane + Cfg::col_s(t);
    const uint32_t tO = t_lane + Cfg::col_o(t);
    const float sl2 = a.scale_log2;
    const float NEG_INF = __int_as_float(0xff800000);
    uint32_t step = 0;
    uint32_t q_rounds = 0;  // kQT: Q loads of this tile consumed
    bool ok = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
      const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
      if (item >= n_eff) break;  // only in the last, partial round
      int bh, pair, split = 0;
      if constexpr (VAR && COMPACT) {
        int b, h;
        sched_decode(sched, a.n_seq, a.n_pairs, a.g.H, CAUSAL, true, item, b, h, pair);
        bh = b * a.g.H + h;
      } else if constexpr (SPLIT) {
        bh = item / a.splits;
        split = item - bh * a.splits;
        pair = 0;
      } else {
        decode_item(item, a, CAUSAL, bh, pair);
      }
      const int qt = 2 * pair + t;
      int J;
      int key_lim = 0;  // VAR: the last key this row may see, relative to the sequence
      int t0 = 0;       // SPLIT: the split's first key tile
      int Jpair = 0;    // kQT: steps of the pair (Q is loaded when > 0)
      if constexpr (VAR) {
        const Seq sq = seq_of<KLENS>(bh, a.g);
        J = var_tile_steps(qt, sq, CAUSAL);
        if constexpr (kQT) Jpair = max(J, var_tile_steps(2 * pair + 1 - t, sq, CAUSAL));
        key_lim = sq.nk - 1;
        if (CAUSAL) key_lim = min(key_lim, qt * kTile + r + sq.nk - sq.nq);
        if constexpr (SPLIT) {
          int t1;
          Jpair = split_tiles(a, split, Jpair, t1);  // the longer tile bounds both
          J = split_tiles(a, split, J, t0);
          const int row = qt * kTile + r;
          if (J == 0 && row < sq.nq) {  // a split past the keys weighs nothing in the merge
            const size_t part = (static_cast<size_t>(bh) * a.splits + split) * a.nq_pad + row;
            float4* po = reinterpret_cast<float4*>(a.part_o + part * D);
            for (int c = 0; c < D / 4; ++c) po[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            a.part_lse[part] = NEG_INF;
          }
        }
      } else {
        J = tile_steps(qt, a, CAUSAL);
        if constexpr (kQT) Jpair = max(J, tile_steps(2 * pair + 1 - t, a, CAUSAL));
      }
      if constexpr (kQT) {
        // Q_t was loaded for this item when either tile of the pair has steps;
        // copy row r into TMEM (bf16 pairs, as P is stored), release Q's
        // buffer, and tell the MMA warp when this tile will use it. The S
        // products of the previous item read the old copy: every one of them
        // completed before this warpgroup's waits on s_full returned.
        if (Jpair > 0) {
          ok = mbar_wait_warp(smem_u32(&bars->q_full[t]), q_rounds & 1, abort, a.status);
          if (!ok) break;
          ++q_rounds;
          if (J > 0) {
            const uint32_t qrow = sQ + t * Cfg::kColBlocks * kBlockBytes + r * 128;
#pragma unroll
            for (int half = 0; half < D / 32; ++half) {  // 16 columns at a time
              uint32_t qw[16];
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const int ch = 4 * half + c4;
                uint4 v;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                             : "r"(qrow + ((ch ^ (r & 7)) << 4)));
                qw[4 * c4] = v.x;
                qw[4 * c4 + 1] = v.y;
                qw[4 * c4 + 2] = v.z;
                qw[4 * c4 + 3] = v.w;
              }
              tmem_st16(t_lane + Cfg::col_q(t) + 16 * half, qw);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&bars->q_empty[t]));
            if (J > 0) mbar_arrive(smem_u32(&bars->q_tmem[t]));
          }
        }
      }
      if (J == 0) continue;
      float m = NEG_INF, l = 0.f;
      for (int j = 0; j < J; ++j) {
        ok = mbar_wait_warp(smem_u32(&bars->s_full[t]), step & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128(tS, sr);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        // masks: causal diagonal tile, and keys past N in the last tile
        int lim = 127;
        if constexpr (VAR) {  // keys past the row's causal limit or past the sequence
          lim = min(lim, key_lim - (t0 + j) * kTile);
        } else {
          if (CAUSAL && j == qt) lim = r;
          if (j == a.n_tiles - 1) lim = min(lim, a.N - 1 - j * kTile);
        }
        const bool masked = lim < 127;
        if (masked) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c > lim) ? NEG_INF : s[c];
        }
        // row max: 8 independent chains of 3-input max
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = fmaxf(s[u], s[u + 8]);
#pragma unroll
        for (int c = 16; c < 128; c += 16) {
#pragma unroll
          for (int u = 0; u < 8; ++u) mx[u] = fmax3(mx[u], s[c + u], s[c + 8 + u]);
        }
        const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                               fmaxf(mx[6], mx[7]));
        float m_use = m, alpha = 1.f;
        bool grow = false;
        if (j == 0) {
          m_use = mt;
        } else if ((mt - m) * sl2 > kRescaleTauLog2) {
          m_use = mt;
          alpha = ex2_approx((m - mt) * sl2);
          grow = true;
        }
        // p = 2^(s * scale*log2e - m * scale*log2e), two lanes per instruction
        const float2 sl2v = make_float2(sl2, sl2);
        // Masked scores are already -inf, so they give 2^-inf = 0 without a
        // select in the loop below (selects there cost 12% of the forward at
        // d = 128 and 20% at d = 64). A row that has seen no key yet keeps
        // m = -inf; 0 in its place keeps its arguments -inf instead of NaN.
        const float m_safe = m_use == NEG_INF ? 0.f : m_use;
        const float2 negv = make_float2(-m_safe * sl2, -m_safe * sl2);
        uint32_t pk[64];
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sl2v, negv);
          float p0, p1;
          if ((c & 7) < kPolyExpPairsPer8) {
            const float2 e = exp2_poly2(x);
            p0 = e.x;
            p1 = e.y;
          } else {
            p0 = ex2_approx(x.x);
            p1 = ex2_approx(x.y);
          }
          acc[c & 3] = fadd2(acc[c & 3], make_float2(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
        const float2 a03 = fadd2(a01, a23);
        l = alpha * l + (a03.x + a03.y);
        tmem_st64(tS, pk);
        if (__any_sync(0xffffffffu, grow)) {
          // O_t still holds the sum up to tile j-1; PV(j-1) completed before S(j) did
          ok = mbar_wait_warp(smem_u32(&bars->o_done[t]), (step - 1) & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            tmem_st32(tO + cc * 32, o);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[t]));
        m = m_use;
        ++step;
      }
      if (!ok) break;
      // epilogue: O / l in bf16 and the log-sum-exp
      ok = mbar_wait_warp(smem_u32(&bars->o_done[t]), (step - 1) & 1, abort, a.status);
      if (!ok) break;
      tc_fence_after();
      const int row = qt * kTile + r;
      bool store;
      float inv_l;
      __nv_bfloat16* orow;
      Seq sq;
      if constexpr (VAR) {  // a row that saw no key has l = 0: O = 0, LSE = -inf
        sq = seq_of<KLENS>(bh, a.g);
        store = row < sq.nq;
        inv_l = l > 0.f ? 1.f / l : 0.f;
        orow = a.o + sq.bb * a.so.batch + sq.hh * a.so.head +
               static_cast<int64_t>(sq.q0 + row) * a.so.row;
#ifdef FA_DEBUG  // the batch coordinates span 1 (packed) or the B sequences (dense)
        if (store)
          store = fa_dcheck(in_span(a.so, a.g.cu_q != nullptr ? 1 : a.BH / a.g.H, a.g.H,
                                    a.g.rows_q, D, orow - a.o, D) &&
                                FA_IN_RANGE(sq.q0 + row, a.g.rows_q),
                            a.status);
#endif
      } else {
        store = row < a.N;
        inv_l = 1.f / l;
        orow = a.o + (bh / a.H) * a.so.batch + (bh % a.H) * a.so.head +
               static_cast<int64_t>(row) * a.so.row;
#ifdef FA_DEBUG
        if (store) store = fa_dcheck(in_span(a.so, a.BH / a.H, a.H, a.N, D, orow - a.o, D), a.status);
#endif
      }
      if constexpr (SPLIT) {  // the split's normalised rows and log2 LSE, fp32
        const size_t part = (static_cast<size_t>(bh) * a.splits + split) * a.nq_pad + row;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          if (store) {
            float4* po = reinterpret_cast<float4*>(a.part_o + part * D + cc * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              po[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv_l, __uint_as_float(o[4 * v4 + 1]) * inv_l,
                                   __uint_as_float(o[4 * v4 + 2]) * inv_l,
                                   __uint_as_float(o[4 * v4 + 3]) * inv_l);
          }
        }
        if (store)
          a.part_lse[part] = l > 0.f ? fmaf(m, a.scale * 1.4426950408889634f, lg2_approx(l)) : NEG_INF;
        continue;
      }
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * v4 + 0]) * inv_l, __uint_as_float(o[8 * v4 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv_l, __uint_as_float(o[8 * v4 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv_l, __uint_as_float(o[8 * v4 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv_l, __uint_as_float(o[8 * v4 + 7]) * inv_l);
            dst[v4] = w;
          }
        }
      }
      if constexpr (VAR) {
        if (store)
          a.lse[static_cast<size_t>(sq.bb * a.g.H + sq.hh) * a.g.rows_q + sq.q0 + row] =
              l > 0.f ? fmaf(m, a.scale, lg2_approx(l) * 0.69314718055994531f)
                      : __int_as_float(0xff800000);
      } else {
        if (store)
          a.lse[static_cast<size_t>(bh) * a.N + row] =
              fmaf(m, a.scale, lg2_approx(l) * 0.69314718055994531f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int D, bool CAUSAL, bool VAR = false, bool COMPACT = false, bool KLENS = false,
          bool SPLIT = false>
cudaError_t launch_fwd_t(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const typename FwdArgsSel<VAR, SPLIT>::type& a,
                         cudaStream_t stream, int extra_smem = 0) {
  const int smem = fwd_smem_bytes<D>() + extra_smem;
  auto kern = fwd_kernel<D, CAUSAL, VAR, COMPACT, KLENS, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = min(a.n_items, p.num_sms);
  kern<<<grid, kFwdThreads, smem, stream>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

template <int D>
cudaError_t launch_var_d(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const FwdVarArgs& a, cudaStream_t stream,
                         int extra) {
  if (a.compact)
    return p.causal ? launch_fwd_t<D, true, true, true>(p, mq, mk, mv, a, stream, extra)
                    : launch_fwd_t<D, false, true, true>(p, mq, mk, mv, a, stream, extra);
  if (p.klens)  // dense batch with per-sequence key counts
    return p.causal ? launch_fwd_t<D, true, true, false, true>(p, mq, mk, mv, a, stream)
                    : launch_fwd_t<D, false, true, false, true>(p, mq, mk, mv, a, stream);
  return p.causal ? launch_fwd_t<D, true, true>(p, mq, mk, mv, a, stream)
                  : launch_fwd_t<D, false, true>(p, mq, mk, mv, a, stream);
}

cudaError_t launch_fwd_var(const Problem& p, const void* q, const void* k, const void* v,
                           void* o, float* lse, cudaStream_t stream) {
  const bool packed = p.cu_q != nullptr;
  const int planes_b = packed ? 1 : p.B;
  CUtensorMap mq, mk, mv;
  if (!make_tile_map(&mq, q, planes_b, p.H, p.rows_q, p.d, p.st[kQ]) ||
      !make_tile_map(&mk, k, planes_b, p.H, p.rows_k, p.d, p.st[kK]) ||
      !make_tile_map(&mv, v, planes_b, p.H, p.rows_k, p.d, p.st[kV]))
    return cudaErrorInvalidValue;
  FwdVarArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = p.status;
  a.BH = p.B * p.H;
  a.n_pairs = ((p.max_q + kTile - 1) / kTile + 1) / 2;
  a.n_items = a.BH * a.n_pairs;
  a.scale = p.scale;
  a.scale_log2 = clamped_scale_log2(p.scale);
  a.so = p.st[kO];
  a.g = VarGeom{p.cu_q, p.cu_k, p.H, p.N, p.Nk, p.rows_q, p.rows_k, p.max_q, p.max_k};
  a.n_seq = p.B;
  // the schedule's arrays after the barriers (their size rounded up to 16
  // bytes), if they fit in the shared memory the kernel leaves spare
  const size_t sched_bytes = 16 + 4 * sched_ints(p.B, a.n_pairs);
  const size_t base_bytes = p.d <= 32 ? fwd_smem_bytes<32>() : p.d <= 64 ? fwd_smem_bytes<64>()
                          : p.d <= 96 ? fwd_smem_bytes<96>() : fwd_smem_bytes<128>();
  // the builder's per-warp counters (P + 1 ints per warp, at least one warp)
  // go into the K/V ring
  const int ring_ints = (p.d <= 32 ? FwdCfg<32>::kRingBytes : p.d <= 64 ? FwdCfg<64>::kRingBytes
                         : p.d <= 96 ? FwdCfg<96>::kRingBytes : FwdCfg<128>::kRingBytes) / 4;
  a.compact = packed && base_bytes + sched_bytes <= 232448 && a.n_pairs + 1 <= ring_ints;
  const int extra = a.compact ? static_cast<int>(sched_bytes) : 0;
  switch (p.d) {
    case 32:
      return launch_var_d<32>(p, mq, mk, mv, a, stream, extra);
    case 64:
      return launch_var_d<64>(p, mq, mk, mv, a, stream, extra);
    case 96:
      return launch_var_d<96>(p, mq, mk, mv, a, stream, extra);
    default:
      return launch_var_d<128>(p, mq, mk, mv, a, stream, extra);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_split_d(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const FwdSplitArgs& a, cudaStream_t stream) {
  return p.klens ? launch_fwd_t<D, CAUSAL, true, false, true, true>(p, mq, mk, mv, a, stream)
                 : launch_fwd_t<D, CAUSAL, true, false, false, true>(p, mq, mk, mv, a, stream);
}

bool fwd_split_supported(int d) { return d == 64 || d == 128; }

cudaError_t launch_fwd_split(const Problem& p, const void* q, const void* k, const void* v,
                             float* part_o, float* part_lse, int splits, int nq_pad,
                             cudaStream_t stream) {
  if (!fwd_split_supported(p.d) || p.cu_q != nullptr || p.max_q > kTile) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  if (!make_tile_map(&mq, q, p.B, p.H, p.rows_q, p.d, p.st[kQ]) ||
      !make_tile_map(&mk, k, p.B, p.H, p.rows_k, p.d, p.st[kK]) ||
      !make_tile_map(&mv, v, p.B, p.H, p.rows_k, p.d, p.st[kV]))
    return cudaErrorInvalidValue;
  FwdSplitArgs a;
  a.o = nullptr;
  a.lse = nullptr;
  a.status = p.status;
  a.BH = p.B * p.H;
  a.n_pairs = 1;
  a.n_items = a.BH * splits;
  a.n_seq = p.B;
  a.compact = 0;
  a.scale = p.scale;
  a.scale_log2 = clamped_scale_log2(p.scale);
  a.so = p.st[kO];
  a.g = VarGeom{p.cu_q, p.cu_k, p.H, p.N, p.Nk, p.rows_q, p.rows_k, p.max_q, p.max_k};
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.splits = splits;
  a.nq_pad = nq_pad;
  if (p.d == 64)
    return p.causal ? launch_split_d<64, true>(p, mq, mk, mv, a, stream)
                    : launch_split_d<64, false>(p, mq, mk, mv, a, stream);
  return p.causal ? launch_split_d<128, true>(p, mq, mk, mv, a, stream)
                  : launch_split_d<128, false>(p, mq, mk, mv, a, stream);
}

cudaError_t launch_fwd(const Problem& p, const void* q, const void* k, const void* v, void* o,
                       float* lse, cudaStream_t stream) {
  if (p.var) return launch_fwd_var(p, q, k, v, o, lse, stream);
  if (p.d == 256) return launch_fwd256(p, q, k, v, o, lse, stream);
  if (!p.causal && p.d >= 64) {
    // Non-causal at d >= 64 the compile-time-flagged instantiation ran faster
    // on GB300 than the dense one on the same problem, with bit-identical
    // results (B*N = 16384 sweep: +1.5..5.5% at d = 128, +5..8% at d = 96,
    // +1..2% at d = 64; causal and d = 32 were equal or slower): run that one
    // with every sequence of length N.
    Problem pv = p;
    pv.var = 1;
    pv.Nk = p.N;
    pv.rows_q = pv.rows_k = pv.max_q = pv.max_k = p.N;
    return launch_fwd_var(pv, q, k, v, o, lse, stream);
  }
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv;
  if (!make_tile_map(&mq, q, p.B, p.H, p.N, p.d, p.st[kQ]) ||
      !make_tile_map(&mk, k, p.B, p.H, p.N, p.d, p.st[kK]) ||
      !make_tile_map(&mv, v, p.B, p.H, p.N, p.d, p.st[kV]))
    return cudaErrorInvalidValue;
  FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.so = p.st[kO];
  a.H = p.H;
  a.lse = lse;
  a.status = p.status;
  a.N = p.N;
  a.BH = BH;
  a.n_tiles = (p.N + kTile - 1) / kTile;
  a.n_pairs = (a.n_tiles + 1) / 2;
  a.n_items = BH * a.n_pairs;
  a.scale = p.scale;
  a.scale_log2 = clamped_scale_log2(p.scale);
  switch (p.d) {
    case 32:
      return p.causal ? launch_fwd_t<32, true>(p, mq, mk, mv, a, stream)
                      : launch_fwd_t<32, false>(p, mq, mk, mv, a, stream);
    case 64:
      return p.causal ? launch_fwd_t<64, true>(p, mq, mk, mv, a, stream)
                      : launch_fwd_t<64, false>(p, mq, mk, mv, a, stream);
    case 96:
      return p.causal ? launch_fwd_t<96, true>(p, mq, mk, mv, a, stream)
                      : launch_fwd_t<96, false>(p, mq, mk, mv, a, stream);
    default:
      return p.causal ? launch_fwd_t<128, true>(p, mq, mk, mv, a, stream)
                      : launch_fwd_t<128, false>(p, mq, mk, mv, a, stream);
  }
}

}  // namespace fa

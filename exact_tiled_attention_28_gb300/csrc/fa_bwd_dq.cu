// Backward, separate dQ path: a query-stationary kernel that recomputes S and
// dP per tile and accumulates dQ in tensor memory, with no atomics.
//
// What it computes ("Flash Attention v2" notes, "Backward Pass Computation":
// recompute S block by block from Q and K, never materialising N x N
// matrices; the softmax Jacobian is the full one):
//   P_ij = exp(scale q_i.k_j - lse_i),  dS_ij = P_ij (dO_i.v_j - D_i),
//   dQ_i = scale sum_j dS_ij k_j
// with D and the log2-unit lse rows from the backward's pre-pass. The dK/dV
// kernel then runs without its dQ product ("FlashAttention-2 paper" digest,
// "Three changes": work split over query blocks as well as key blocks; here
// the dQ sum over key blocks is owned by one CTA per query block instead of
// being reduced with atomics). The price is two more products per tile
// (S and dP are computed by both kernels): 7 instead of 5.
//
// GB300 mapping:
//  - persistent CTAs over (batch*head, 128-row query block i); causal items
//    longest first (block i visits key blocks 0..i);
//  - warp 8 loads Q_i and dO_i once per item, and streams K_j, V_j through a
//    ring of 128-row slots in the order the products consume them;
//  - warp 9 issues tcgen05.mma, per key block j:
//      S = Q_i K_j^T  and  dP = dO_i V_j^T          (SS, M = 128 queries)
//      dQ += dS K_j                                  (A = dS from TMEM)
//    in the order dQ(j), dP(j+1), S(j+2), so that the tensor core computes the
//    next products while the compute warps turn S and dP into dS;
//  - warps 0-7: two warpgroups, one thread per query row (TMEM lane), each
//    owning 64 of the 128 key columns. lse and D are per-row scalars here.
//    They write dS as packed bf16 over the first 32 of their own S columns,
//    and at the end of an item read dQ out of TMEM and store bf16 dq once.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256) (S double-buffered), dP
// [256,384), dQ [384, 384+d).

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "schedule.cuh"

namespace fa {
namespace {

constexpr int kDqThreads = 320;  // 8 compute warps + load warp + MMA warp
constexpr int kDqLoadWarp = 8;
constexpr int kDqMmaWarp = 9;
constexpr uint32_t kDqTmemCols = 512;
constexpr int kDqBlk = kTile * 64 * 2;  // one 128-row x 64-column bf16 block: 16 KiB
constexpr uint32_t kColDpSep = 256, kColDqSep = 384;

template <int D>
struct DqCfg {
  static_assert(D == 64 || D == 128, "the separate dQ kernel takes d = 64 or 128");
  static constexpr int kColBlocks = D / 64;
  static constexpr int kTileBytes = kTile * kColBlocks * 64 * 2;
  // ring slots of one 128-row K or V tile: K_j and V_j take consecutive
  // slots. S(j+2) is issued right after dQ(j), the last reader of K_j; with
  // 5 slots (d = 128) K_{j+2} goes into the slot V_{j-1} freed, so its copy
  // never waits for dQ(j)
  static constexpr int kSlots = D == 128 ? 5 : 10;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTileBytes;
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffBars = kOffRing + kSlots * kTileBytes;
  __device__ static constexpr uint32_t col_s(uint32_t b) { return 128u * b; }
};

struct DqBarriers {
  uint64_t qd_full, qd_empty;
  uint64_t kv_full[10], kv_empty[10];
  uint64_t s_full[2], dp_full, ds_ready, dq_full, dq_free, drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
constexpr int dq_smem_bytes() {
  return 1024 + DqCfg<D>::kOffBars + static_cast<int>(sizeof(DqBarriers));
}
static_assert(dq_smem_bytes<128>() <= 232448, "dQ kernel shared memory over the sm_103a limit");
static_assert(dq_smem_bytes<64>() <= 232448, "dQ kernel shared memory over the sm_103a limit");

__device__ __forceinline__ void decode_q_item(int item, const BwdDqArgs& a, bool causal, int& bh,
                                              int& i) {
  if (causal) {  // longest first: the last query blocks of every head come first
    i = a.n_tiles - 1 - item / a.BH;
    bh = item % a.BH;
  } else {  // the query blocks of one head adjacent: K and V shared through L2
    bh = item / a.n_tiles;
    i = item % a.n_tiles;
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const BwdDqArgs a) {
  using Cfg = DqCfg<D>;
  constexpr int R = Cfg::kSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + Cfg::kOffQ, sdO = sbase + Cfg::kOffDO, sRing = sbase + Cfg::kOffRing;
  DqBarriers* bars = reinterpret_cast<DqBarriers*>(smem + Cfg::kOffBars);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->qd_full), 1);
    mbar_init(smem_u32(&bars->qd_empty), 1);
    for (int s = 0; s < R; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full[0]), 1);
    mbar_init(smem_u32(&bars->s_full[1]), 1);
    mbar_init(smem_u32(&bars->dp_full), 1);
    mbar_init(smem_u32(&bars->ds_ready), 8);  // one elected lane per compute warp
    mbar_init(smem_u32(&bars->dq_full), 1);
    mbar_init(smem_u32(&bars->dq_free), 8);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kDqMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kDqTmemCols);
    tmem_relinquish();
  }
  if (warp == kDqLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kDqLoadWarp) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();  // Q_i, dO_i: read by this CTA only
      const uint64_t pol_kv = policy_evict_last();  // K_j, V_j: read by every query block
      uint32_t slot_it = 0, q_round = 0;
      bool ok = true;
      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= a.n_items) break;  // only in the last, partial round
        int bh, i;
        decode_q_item(item, a, CAUSAL, bh, i);
        const int hh = bh % a.H, bb = bh / a.H;
        const int J = CAUSAL ? i + 1 : a.n_tiles;
        ok = mbar_wait(smem_u32(&bars->qd_empty), (q_round & 1) ^ 1, abort, a.status);
        if (!ok) break;
        {
          const uint32_t bar = smem_u32(&bars->qd_full);
          mbar_arrive_expect_tx(bar, 2 * Cfg::kTileBytes);
          for (int cb = 0; cb < Cfg::kColBlocks; ++cb) {
            tma_load_4d(sQ + cb * kDqBlk, &tmQ, bar, 64 * cb, i * kTile, hh, bb, pol_q);
            tma_load_4d(sdO + cb * kDqBlk, &tmdO, bar, 64 * cb, i * kTile, hh, bb, pol_q);
          }
          ++q_round;
        }
        for (int j = 0; j < J && ok; ++j) {
          for (int w = 0; w < 2; ++w) {  // K_j then V_j
            const uint32_t s = slot_it % R;
            ok = mbar_wait(smem_u32(&bars->kv_empty[s]), ((slot_it / R) & 1) ^ 1, abort,
                           a.status);
            if (!ok) break;
            const uint32_t bar = smem_u32(&bars->kv_full[s]);
            mbar_arrive_expect_tx(bar, Cfg::kTileBytes);
            for (int cb = 0; cb < Cfg::kColBlocks; ++cb)
              tma_load_4d(sRing + s * Cfg::kTileBytes + cb * kDqBlk, w ? &tmV : &tmK, bar, 64 * cb,
                          j * kTile, hh, bb, pol_kv);
            ++slot_it;
          }
        }
      }
      // Producer tail. Normal path: wait until the consumer has released every
      // slot, so that no barrier arrival lands after the CTA exits. After an
      // abort: wait (bounded) for the copies already issued to land.
      const uint32_t n = min(slot_it, static_cast<uint32_t>(R));
      for (uint32_t u = slot_it - n; u < slot_it; ++u) {
        const uint32_t s = u % R, ph = (u / R) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->kv_empty[s]), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->kv_full[s]), ph, 100000000ull);
      }
      if (q_round > 0) {
        const uint32_t ph = (q_round - 1) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->qd_empty), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->qd_full), ph, 100000000ull);
      }
    }
  } else if (warp == kDqMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // S = Q K^T, dP = dO V^T: M = 128 queries, N = 128 keys, both K-major
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kTile, kTile, false, false);
      // dQ += dS K: A = dS from TMEM, B = K_j MN-major (keys x d), N = d
      constexpr uint32_t idesc_dq = idesc_bf16_f32(kTile, D, false, true);
      uint32_t slot_it = 0, q_round = 0, step = 0, n_done = 0;
      bool ok = true;

      auto issue_qk = [&](uint32_t dst, uint32_t a_tile, uint32_t slot) {
        const SmemDesc da = make_desc_sw128(opaque_u32(a_tile), 16, 1024);
        const SmemDesc db = make_desc_sw128(opaque_u32(sRing + slot * Cfg::kTileBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kDqBlk + (kk & 3) * 32;
          mma_ss(dst, desc_at(da, off), desc_at(db, off), idesc_qk, kk > 0);
        }
      };
      // keys 16kk..16kk+15 of dS sit in the half written by compute warpgroup
      // kk / 4, at column 64 (kk/4) + 8 (kk%4) of the S buffer
      auto issue_dq = [&](uint32_t s_col, uint32_t slot, bool accumulate) {
        const SmemDesc db =
            make_desc_sw128(opaque_u32(sRing + slot * Cfg::kTileBytes), kDqBlk, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(tmem + kColDqSep, tmem + s_col + 64 * (kk >> 2) + 8 * (kk & 3),
                 desc_at(db, kk * 2048), idesc_dq, (accumulate || kk > 0) ? 1u : 0u);
      };
      auto slot_wait = [&](uint32_t idx) {
        return mbar_wait(smem_u32(&bars->kv_full[idx % R]), (idx / R) & 1, abort, a.status);
      };

      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= a.n_items) break;
        int bh, i;
        decode_q_item(item, a, CAUSAL, bh, i);
        const int J = CAUSAL ? i + 1 : a.n_tiles;
        const uint32_t base = slot_it;  // slot index of K_j: base + 2j; of V_j: base + 2j + 1
        ok = mbar_wait(smem_u32(&bars->qd_full), q_round & 1, abort, a.status);
        if (!ok) break;
        // prologue: S(0), dP(0), S(1)
        ok = slot_wait(base);
        if (!ok) break;
        tc_fence_after();
        issue_qk(tmem + Cfg::col_s(step & 1), sQ, base % R);
        mma_commit(smem_u32(&bars->s_full[step & 1]));
        ok = slot_wait(base + 1);
        if (!ok) break;
        tc_fence_after();
        issue_qk(tmem + kColDpSep, sdO, (base + 1) % R);
        mma_commit(smem_u32(&bars->dp_full));
        mma_commit(smem_u32(&bars->kv_empty[(base + 1) % R]));
        if (J == 1) mma_commit(smem_u32(&bars->qd_empty));
        if (J > 1) {
          ok = slot_wait(base + 2);
          if (!ok) break;
          tc_fence_after();
          issue_qk(tmem + Cfg::col_s((step + 1) & 1), sQ, (base + 2) % R);
          mma_commit(smem_u32(&bars->s_full[(step + 1) & 1]));
        }
        for (int u = 0; u < J && ok; ++u, ++step) {
          const uint32_t sb = Cfg::col_s(step & 1);
          ok = mbar_wait(smem_u32(&bars->ds_ready), step & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
          if (u == 0 && n_done > 0) {  // the previous item's dQ has been read out
            ok = mbar_wait(smem_u32(&bars->dq_free), (n_done - 1) & 1, abort, a.status);
            if (!ok) break;
            tc_fence_after();
          }
          issue_dq(sb, (base + 2 * u) % R, u > 0);  // dQ (+)= dS(u) K_u
          mma_commit(smem_u32(&bars->kv_empty[(base + 2 * u) % R]));
          if (u + 1 < J) {  // dP(u+1): the compute warps have read dP(u)
            ok = slot_wait(base + 2 * u + 3);
            if (!ok) break;
            tc_fence_after();
            issue_qk(tmem + kColDpSep, sdO, (base + 2 * u + 3) % R);
            mma_commit(smem_u32(&bars->dp_full));
            mma_commit(smem_u32(&bars->kv_empty[(base + 2 * u + 3) % R]));
            if (u + 2 == J) mma_commit(smem_u32(&bars->qd_empty));  // last reader of Q and dO
          }
          if (u + 2 < J) {  // S(u+2) into this S buffer, after dQ(u) has read dS(u)
            ok = slot_wait(base + 2 * u + 4);
            if (!ok) break;
            tc_fence_after();
            issue_qk(tmem + sb, sQ, (base + 2 * u + 4) % R);
            mma_commit(smem_u32(&bars->s_full[step & 1]));
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->dq_full));
        ++n_done;
        ++q_round;
        slot_it = base + 2 * J;
      }
      // every MMA issued so far completes before TMEM is released
      mma_commit(smem_u32(&bars->drain));
      mbar_drain(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else {
    // ------------------------------- compute warps: P, dS; the dQ epilogue
    const int wg = warp >> 2;              // key columns 64 wg .. 64 wg + 63
    const int r = (warp & 3) * 32 + lane;  // query row within the block = TMEM lane
    const uint32_t t_lane = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16);
    const float sl2 = a.scale_log2;
    uint32_t step = 0, n_done = 0;
    bool ok = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
      const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
      if (item >= a.n_items) break;
      int bh, i;
      decode_q_item(item, a, CAUSAL, bh, i);
      const int J = CAUSAL ? i + 1 : a.n_tiles;
      const int row = i * kTile + r;
      // pad rows (row >= N) hold lse2 = +inf, D = 0: their P and dS are 0
      const size_t prow = static_cast<size_t>(bh) * a.Npad + row;
      const float lse2 = a.lse2[prow];
      const float Dr = a.Drow[prow];
      const int kcol0 = 64 * wg;
      for (int u = 0; u < J; ++u, ++step) {
        const uint32_t tS = t_lane + Cfg::col_s(step & 1) + kcol0;
        ok = mbar_wait_warp(smem_u32(&bars->s_full[step & 1]), (step >> 1) & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64(tS, sr);
        const bool diag = CAUSAL && u == i;  // key columns above the row are masked
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x = ffma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])),
                                 make_float2(sl2, sl2), make_float2(-lse2, -lse2));
          float p0 = ex2_approx(x.x);
          float p1 = ex2_approx(x.y);
          if (diag) {
            p0 = (kcol0 + 2 * c > r) ? 0.f : p0;
            p1 = (kcol0 + 2 * c + 1 > r) ? 0.f : p1;
          }
          pk[c] = pack_bf16x2(p0, p1);
        }
        ok = mbar_wait_warp(smem_u32(&bars->dp_full), step & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dp[32];
          tmem_ld32(t_lane + kColDpSep + kcol0 + 32 * h, dp);
          uint32_t ds[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 pf =
                __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[16 * h + c]));
            const float2 g = fadd2(make_float2(__uint_as_float(dp[2 * c]), __uint_as_float(dp[2 * c + 1])),
                                   make_float2(-Dr, -Dr));
            const float2 v = fmul2(pf, g);
            ds[c] = pack_bf16x2(v.x, v.y);
          }
          tmem_st16(tS + 16 * h, ds);  // over S columns this warpgroup has read
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->ds_ready));
      }
      if (!ok) break;
      // epilogue: warpgroup wg reads dQ columns wg*d/2 .. and stores them
      ok = mbar_wait_warp(smem_u32(&bars->dq_full), n_done & 1, abort, a.status);
      if (!ok) break;
      tc_fence_after();
      constexpr int kHalf = D / 2;
      uint32_t v[kHalf];
#pragma unroll
      for (int c0 = 0; c0 < kHalf; c0 += 32) {
        uint32_t t32[32];
        tmem_ld32(t_lane + kColDqSep + wg * kHalf + c0, t32);
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c0 + c] = t32[c];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
      const int64_t off = (bh / a.H) * a.sdq.batch + (bh % a.H) * a.sdq.head +
                          static_cast<int64_t>(row) * a.sdq.row + wg * kHalf;
      if (row < a.N && fa_dcheck(FA_IN_SPAN(a.sdq, a.BH / a.H, a.H, a.N, D, off, kHalf), a.status)) {
        uint4* dst = reinterpret_cast<uint4*>(a.dq + off);
        const float sc = a.scale;
#pragma unroll
        for (int v4 = 0; v4 < kHalf / 8; ++v4) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[8 * v4 + 0]) * sc, __uint_as_float(v[8 * v4 + 1]) * sc);
          w.y = pack_bf16x2(__uint_as_float(v[8 * v4 + 2]) * sc, __uint_as_float(v[8 * v4 + 3]) * sc);
          w.z = pack_bf16x2(__uint_as_float(v[8 * v4 + 4]) * sc, __uint_as_float(v[8 * v4 + 5]) * sc);
          w.w = pack_bf16x2(__uint_as_float(v[8 * v4 + 6]) * sc, __uint_as_float(v[8 * v4 + 7]) * sc);
          dst[v4] = w;
        }
      }
      ++n_done;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kDqMmaWarp) tmem_dealloc(tmem, kDqTmemCols);
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const Problem& p, const CUtensorMap* maps, const BwdDqArgs& a,
                     cudaStream_t stream) {
  constexpr int smem = dq_smem_bytes<D>();
  auto kern = bwd_dq_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = min(a.n_items, p.num_sms);
  kern<<<grid, kDqThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], a);
  return cudaGetLastError();
}

}  // namespace

bool bwd_dq_separate_supported(int d) { return d == 64 || d == 128; }

cudaError_t launch_bwd_dq_separate(const Problem& p, const CUtensorMap* maps, const BwdDqArgs& a,
                                   cudaStream_t stream) {
  if (p.d == 64)
    return p.causal ? launch_t<64, true>(p, maps, a, stream) : launch_t<64, false>(p, maps, a, stream);
  if (p.d == 128)
    return p.causal ? launch_t<128, true>(p, maps, a, stream)
                    : launch_t<128, false>(p, maps, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa

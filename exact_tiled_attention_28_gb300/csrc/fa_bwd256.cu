// dK / dV stage of the backward at head dimension 256 ("Flash Attention v2"
// notes, "Detailed Differences", 3 "Head Dimension Support": the tiled method
// up to head_dim = 256; "Backward Pass Computation": recompute S and P per
// block, then dP, dS and the three gradients).
//
// The d <= 128 kernel keeps dK_j and dV_j of a 128-key block in TMEM with
// the keys as MMA rows; at d = 256 those two alone would fill all 512 TMEM
// columns. Here a work item is a block of 64 keys, the MMAs run with the 128
// queries of a block (or 128 head-dim rows) as M, and the key-side gradients
// are kept transposed, head-dim rows by key columns, in two d-halves:
//
//   S    = Q_i K_j^T             M = 128 queries, N = 64 keys, K = 256
//   dP   = dO_i V_j^T            the same
//   P    = exp2(S scale log2e - lse2_i), dS = P (dP - D_i)     (compute warps)
//   dV^T[h] += dO_i^T[h] P       M = 128 head dims of half h, N = 64, K = 128 queries
//   dK^T[h] += Q_i^T[h] dS       the same
//   dQ_i^T[h] = K_j^T[h] dS^T    M = 128 head dims, N = 128 queries, K = 64 keys
//
// TMEM (512 columns): S [0,64), dP [64,128), dQ^T half [128,256), dV^T
// [256,384) and dK^T [384,512) as two 64-column halves each. The dQ^T halves
// go through their one buffer in turn; four read-out warps add each to the
// fp32 accumulator (a warp's 32 lanes are 32 consecutive head dims of one
// query row: one 128-byte segment per reduction).
//
// Shared memory (224 KiB + rows): Q_i and dO_i (128 x 256 bf16 each), K_j and
// V_j (64 x 256 each), P and dS (128 x 64 each, written by the compute warps
// in the 128-byte swizzled layout the MMAs read), the lse2 and D rows of
// block i. There is room for one Q_i / dO_i buffer only. Non-causal, the dK
// MMAs run first and release Q_i, whose successor the next block's S needs
// first, and dO_i follows after the dV MMAs; causal keeps dV first (measured
// marginally faster). Both copies overlap the dQ^T MMAs.
//
// 512 threads: warp 0 TMA loader, warp 1 MMA issuer, warps 4-7 compute (one
// thread per query row = TMEM lane), warps 8-15 dQ^T read-out and the dK /
// dV epilogue (one thread per head-dim row; warps 8-11 take query columns
// 0-63 of each dQ^T half and head-dim half 0 of dK / dV, warps 12-15 the
// rest). The read-out is the kernel's critical path: a dQ^T half's next
// product waits for it, and each read-out warp's reductions issue one by
// one, so eight warps halve it. Launched at 128 registers a thread, the
// warpgroups rebalance with setmaxnreg: loader / MMA 96, compute 160,
// read-out 128 (per SM sub-partition 96 + 160 + 128 + 128 = 512, the launch
// total). Persistent, one CTA per SM; every barrier wait is bounded.

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "schedule.cuh"

namespace fa {
namespace {

constexpr int kKeys = 64;                 // keys per work item
constexpr int kThreadsB = 512;
constexpr int kLoadWarpB = 0;
constexpr int kMmaWarpB = 1;
constexpr int kComputeWarp0 = 4;
constexpr int kDqWarp0 = 8;
constexpr int kQBlk = kTile * 64 * 2;     // 16 KiB: 128 rows x 64 columns
constexpr int kKBlk = kKeys * 64 * 2;     // 8 KiB: 64 rows x 64 columns
constexpr int kPBytes = kTile * kKeys * 2;  // 16 KiB: 128 query rows x 64 keys
constexpr int kOffQ = 0;
constexpr int kOffDO = kOffQ + 4 * kQBlk;
constexpr int kOffK = kOffDO + 4 * kQBlk;
constexpr int kOffV = kOffK + 4 * kKBlk;
constexpr int kOffP = kOffV + 4 * kKBlk;
constexpr int kOffDS = kOffP + kPBytes;
constexpr int kOffLse = kOffDS + kPBytes;
constexpr int kOffDrow = kOffLse + kTile * 4;
constexpr int kOffBarsB = kOffDrow + kTile * 4;
constexpr uint32_t kTmemColsB = 512;
constexpr uint32_t kColS = 0, kColDP = 64, kColDQ = 128, kColDV = 256, kColDK = 384;

struct BarsB256 {
  uint64_t kv_full, kv_empty, do_full, do_empty;
  uint64_t q_full[2], q_empty[2];  // Q_i (causal: in two 128-column halves)
  uint64_t s_full, dp_full, pds_ready, pds_free, dq_full, dq_free, acc_done, acc_free, drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int smem_b256_bytes() { return 1024 + kOffBarsB + static_cast<int>(sizeof(BarsB256)); }
static_assert(smem_b256_bytes() <= 232448, "d = 256 backward shared memory over the limit");

// Work item -> (b * H + h, key block j). Causal: key block 0 sees every
// query block, so the blocks go in increasing j (longest first); otherwise
// the key blocks of one head are adjacent, so that concurrent CTAs stream
// the same Q_i / dO_i through L2.
__device__ __forceinline__ void decode_b256(int item, const Bwd256Args& a, bool causal, int& bh,
                                            int& j) {
  if (causal) {
    j = item / a.BH;
    bh = item % a.BH;
  } else {
    bh = item / a.n_kb;
    j = item % a.n_kb;
  }
}

// First query block key block j meets: the causal diagonal (query i sees
// keys <= i) puts keys 64 j .. 64 j + 63 in query blocks from 64 j / 128 on.
__device__ __forceinline__ int first_qblock(int j, bool causal) { return causal ? j >> 1 : 0; }

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd256_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO, const Bwd256Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kQParts = CAUSAL ? 2 : 1;  // copies (and barriers) per Q_i
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sQ = s0 + kOffQ, sDO = s0 + kOffDO, sK = s0 + kOffK, sV = s0 + kOffV;
  const uint32_t sP = s0 + kOffP, sDS = s0 + kOffDS;
  const float* sLse = reinterpret_cast<const float*>(smem + kOffLse);
  const float* sDrow = reinterpret_cast<const float*>(smem + kOffDrow);
  BarsB256* bars = reinterpret_cast<BarsB256*>(smem + kOffBarsB);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->kv_full), 1);
    mbar_init(smem_u32(&bars->kv_empty), 1);
    for (int hq = 0; hq < 2; ++hq) {
      mbar_init(smem_u32(&bars->q_full[hq]), 1);
      mbar_init(smem_u32(&bars->q_empty[hq]), 1);
    }
    mbar_init(smem_u32(&bars->do_full), 1);
    mbar_init(smem_u32(&bars->do_empty), 1);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->dp_full), 1);
    mbar_init(smem_u32(&bars->pds_ready), 4);  // one elected lane per compute warp
    mbar_init(smem_u32(&bars->pds_free), 1);
    mbar_init(smem_u32(&bars->dq_full), 1);
    mbar_init(smem_u32(&bars->dq_free), 8);    // one elected lane per read-out warp
    mbar_init(smem_u32(&bars->acc_done), 1);
    mbar_init(smem_u32(&bars->acc_free), 8);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarpB) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemColsB);
    tmem_relinquish();
  }
  if (warp == kLoadWarpB && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < kComputeWarp0) {
    setmaxnreg_dec<96>();  // all of warps 0-3; 2 and 3 have no role
  if (warp == kLoadWarpB) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      const uint64_t pol_qd = policy_evict_last();   // read by every key block of the head
      const uint64_t pol_kv = policy_evict_first();  // read by one work item
      uint32_t it = 0, g = 0;  // items and query blocks loaded
      bool ok = true;
      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd, ++it) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= a.n_items) break;  // only in the last, partial round
        int bh, j;
        decode_b256(item, a, CAUSAL, bh, j);
        const int hh = bh % a.H, bb = bh / a.H;
        const int i0 = first_qblock(j, CAUSAL);
        if (it > 0) {
          ok = mbar_wait(smem_u32(&bars->kv_empty), (it - 1) & 1, abort, a.status);
          if (!ok) break;
        }
        {
          const uint32_t bar = smem_u32(&bars->kv_full);
          mbar_arrive_expect_tx(bar, 8 * kKBlk);
          tma_load_5d(sK, &tmK, bar, 0, j * kKeys, 0, hh, bb, pol_kv);  // all four column blocks
          tma_load_5d(sV, &tmV, bar, 0, j * kKeys, 0, hh, bb, pol_kv);
        }
        for (int i = i0; i < a.n_qb && ok; ++i, ++g) {
          const size_t row0 = static_cast<size_t>(bh) * a.Npad + static_cast<size_t>(i) * kTile;
          // Causal, Q_i comes in two halves of two column blocks: the dK^T
          // half that reads each releases it, and S's first eight K steps
          // need only the first (measured 3.8% faster causal, 2.6% slower
          // non-causal, which loads Q_i with one copy)
          auto load_q = [&]() {
            for (int hq = 0; hq < kQParts; ++hq) {
              if (g > 0 &&
                  !mbar_wait(smem_u32(&bars->q_empty[hq]), (g - 1) & 1, abort, a.status))
                return false;
              const uint32_t bar = smem_u32(&bars->q_full[hq]);
              mbar_arrive_expect_tx(bar, 4 * kQBlk / kQParts + (hq == 0 ? kTile * 4 : 0));
              tma_load_5d(sQ + 2 * hq * kQBlk, &tmQ, bar, 0, i * kTile, 2 * hq, hh, bb, pol_qd);
              if (hq == 0) cp_bulk_g2s(s0 + kOffLse, a.lse2 + row0, kTile * 4, bar);
            }
            return true;
          };
          auto load_do = [&]() {
            if (g > 0 && !mbar_wait(smem_u32(&bars->do_empty), (g - 1) & 1, abort, a.status))
              return false;
            const uint32_t bar = smem_u32(&bars->do_full);
            mbar_arrive_expect_tx(bar, 4 * kQBlk + kTile * 4);
            tma_load_5d(sDO, &tmDO, bar, 0, i * kTile, 0, hh, bb, pol_qd);
            cp_bulk_g2s(s0 + kOffDrow, a.Drow + row0, kTile * 4, bar);
            return true;
          };
          // the copies follow the order in which the MMAs release the buffers
          ok = CAUSAL ? (load_do() && load_q()) : (load_q() && load_do());
          if (!ok) break;
        }
      }
      // producer tail: the consumers have released everything issued before
      // the CTA exits (after an abort, the copies already issued may land)
      if (it > 0) {
        const uint32_t ph = (it - 1) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->kv_empty), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->kv_full), ph, 100000000ull);
      }
      if (g > 0) {
        const uint32_t ph = (g - 1) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->do_empty), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->do_full), ph, 100000000ull);
        for (int hq = 0; hq < kQParts; ++hq) {
          if (ok) ok = mbar_wait(smem_u32(&bars->q_empty[hq]), ph, abort, a.status);
          if (!ok) mbar_drain(smem_u32(&bars->q_full[hq]), ph, 100000000ull);
        }
      }
    }
  } else if (warp == kMmaWarpB) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kKeys, false, false);
      constexpr uint32_t idesc_g = idesc_bf16_f32(kTile, kKeys, true, true);
      constexpr uint32_t idesc_q = idesc_bf16_f32(kTile, kTile, true, false);
      // S (or dP) = X Y^T over d = 256 in 16-column steps; X: 128 rows in four
      // 64-column blocks (K-major), Y: 64 rows in four blocks (K-major)
      auto issue_s = [&](uint32_t dst, uint32_t x, uint32_t y) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint32_t ox = (kk >> 2) * kQBlk + (kk & 3) * 32;
          const uint32_t oy = (kk >> 2) * kKBlk + (kk & 3) * 32;
          mma_ss(dst, desc_at(make_desc_sw128(opaque_u32(x + ox), 16, 1024), 0),
                 desc_at(make_desc_sw128(opaque_u32(y + oy), 16, 1024), 0), idesc_s, kk > 0);
        }
      };
      // the same over head dims 128 h .. 128 h + 127 (K steps 8 h .. 8 h + 7)
      auto issue_s_half = [&](uint32_t dst, uint32_t x, uint32_t y, int h) {
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
          const int kk = 8 * h + k8;
          const uint32_t ox = (kk >> 2) * kQBlk + (kk & 3) * 32;
          const uint32_t oy = (kk >> 2) * kKBlk + (kk & 3) * 32;
          mma_ss(dst, desc_at(make_desc_sw128(opaque_u32(x + ox), 16, 1024), 0),
                 desc_at(make_desc_sw128(opaque_u32(y + oy), 16, 1024), 0), idesc_s, kk > 0);
        }
      };
      // G^T[h] (+)= X^T[h] Z over the 128 queries in 16-row steps: X (Q or
      // dO) read MN-major, head-dim half h = its column blocks 2h, 2h + 1;
      // Z (P or dS, 128 x 64) read MN-major
      auto issue_g = [&](uint32_t dst, uint32_t x, int h, uint32_t z, bool accumulate) {
        const SmemDesc dx = make_desc_sw128(opaque_u32(x + 2 * h * kQBlk), kQBlk, 1024);
        const SmemDesc dz = make_desc_sw128(opaque_u32(z), kPBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ss(dst, desc_at(dx, kk * 2048), desc_at(dz, kk * 2048), idesc_g,
                 (accumulate || kk > 0) ? 1u : 0u);
      };
      // dQ^T[h] = K^T[h] dS^T over the 64 keys: K read MN-major (column
      // blocks 2h, 2h + 1), dS read K-major (query rows, key columns)
      auto issue_dq = [&](int h) {
        const SmemDesc dk = make_desc_sw128(opaque_u32(sK + 2 * h * kKBlk), kKBlk, 1024);
        const SmemDesc dd = make_desc_sw128(opaque_u32(sDS), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_ss(tmem + kColDQ, desc_at(dk, kk * 2048), desc_at(dd, kk * 32), idesc_q, kk > 0);
      };
      uint32_t it = 0, g = 0;
      bool ok = true;
      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd, ++it) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= a.n_items) break;  // only in the last, partial round
        int bh, j;
        decode_b256(item, a, CAUSAL, bh, j);
        const int i0 = first_qblock(j, CAUSAL);
        ok = mbar_wait(smem_u32(&bars->kv_full), it & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        for (int i = i0; i < a.n_qb && ok; ++i, ++g) {
          const bool first = i == i0;
          ok = mbar_wait(smem_u32(&bars->q_full[0]), g & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
          if constexpr (kQParts == 2) {
            issue_s_half(tmem + kColS, sQ, sK, 0);  // head dims 0-127: Q_i's first half
            ok = mbar_wait(smem_u32(&bars->q_full[1]), g & 1, abort, a.status);
            if (!ok) break;
            tc_fence_after();
            issue_s_half(tmem + kColS, sQ, sK, 1);
          } else {
            issue_s(tmem + kColS, sQ, sK);
          }
          mma_commit(smem_u32(&bars->s_full));  // the compute warps start P while dP runs
          ok = mbar_wait(smem_u32(&bars->do_full), g & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
          issue_s(tmem + kColDP, sDO, sV);
          mma_commit(smem_u32(&bars->dp_full));
          // P and dS written, S and dP read out
          ok = mbar_wait(smem_u32(&bars->pds_ready), g & 1, abort, a.status);
          if (!ok) break;
          if (first && it > 0) {  // the previous item's epilogue has read dK^T, dV^T
            ok = mbar_wait(smem_u32(&bars->acc_free), (it - 1) & 1, abort, a.status);
            if (!ok) break;
          }
          tc_fence_after();
          // non-causal: dK first, so Q_i is released for the next block's
          // copy, which the next block's first MMA (S) waits for; causal
          // measured marginally faster with dV first
          if constexpr (!CAUSAL) {
            issue_g(tmem + kColDK, sQ, 0, sDS, !first);
            issue_g(tmem + kColDK + 64, sQ, 1, sDS, !first);
            mma_commit(smem_u32(&bars->q_empty[0]));
          }
          issue_g(tmem + kColDV, sDO, 0, sP, !first);
          issue_g(tmem + kColDV + 64, sDO, 1, sP, !first);
          mma_commit(smem_u32(&bars->do_empty));
          if constexpr (CAUSAL) {
            issue_g(tmem + kColDK, sQ, 0, sDS, !first);
            mma_commit(smem_u32(&bars->q_empty[0]));
            issue_g(tmem + kColDK + 64, sQ, 1, sDS, !first);
            mma_commit(smem_u32(&bars->q_empty[1]));
          }
          for (int h = 0; h < 2 && ok; ++h) {
            const uint32_t c = 2 * g + h;  // dQ^T halves issued so far
            if (c > 0) {  // the read-out has taken the previous half
              ok = mbar_wait(smem_u32(&bars->dq_free), (c - 1) & 1, abort, a.status);
              if (!ok) break;
              tc_fence_after();
            }
            issue_dq(h);
            mma_commit(smem_u32(&bars->dq_full));
          }
          mma_commit(smem_u32(&bars->pds_free));
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->kv_empty));
        mma_commit(smem_u32(&bars->acc_done));
      }
      // every MMA issued so far completes before TMEM is released
      mma_commit(smem_u32(&bars->drain));
      mbar_drain(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  }
  } else if (warp < kComputeWarp0 + 4) {
    setmaxnreg_inc<160>();
    // ------------------------------------------------------ P and dS rows
    const int r = (warp - kComputeWarp0) * 32 + lane;  // query row = TMEM lane
    const uint32_t t_lane = tmem + ((static_cast<uint32_t>(warp & 3) * 32u) << 16);
    const float sl2 = a.scale_log2;
    uint32_t g = 0;
    bool ok = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
      const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
      if (item >= a.n_items) break;  // only in the last, partial round
      int bh, j;
      decode_b256(item, a, CAUSAL, bh, j);
      const int i0 = first_qblock(j, CAUSAL);
      for (int i = i0; i < a.n_qb; ++i, ++g) {
        // phase A, P = exp2(S scale log2e - lse2), once S is in: it runs
        // while the tensor core computes dP
        ok = mbar_wait_warp(smem_u32(&bars->s_full), g & 1, abort, a.status);
        // the lse2 rows came with Q_i
        if (ok) ok = mbar_wait_warp(smem_u32(&bars->q_full[0]), g & 1, abort, a.status);
        // the MMAs of the previous block have read P and dS
        if (ok && g > 0) ok = mbar_wait_warp(smem_u32(&bars->pds_free), (g - 1) & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        const float l2 = sLse[r];
        // last key column this row keeps: keys past N, and the causal diagonal
        int lim = min(kKeys - 1, a.N - 1 - j * kKeys);
        if (CAUSAL && i == i0) lim = min(lim, i * kTile + r - j * kKeys);
        const uint32_t prow = sP + r * 128, drow = sDS + r * 128;
        // Two copies of the P loop, so that blocks with nothing to mask (all
        // but the diagonal and the last) run no select: selects in the loop
        // cost 12% of the kernel.
        const bool masked = lim < kKeys - 1;
        float pf[64];  // P in fp32, for dS
        auto p_row = [&](int c, const uint32_t (&sv)[32], bool mask, uint32_t (&pk)[16]) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int k0 = 32 * c + 2 * t;
            float p0 = ex2_approx(fmaf(__uint_as_float(sv[2 * t]), sl2, -l2));
            float p1 = ex2_approx(fmaf(__uint_as_float(sv[2 * t + 1]), sl2, -l2));
            if (mask) {
              p0 = k0 > lim ? 0.f : p0;
              p1 = k0 + 1 > lim ? 0.f : p1;
            }
            pf[k0] = p0;
            pf[k0 + 1] = p1;
            pk[t] = pack_bf16x2(p0, p1);
          }
        };
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sv[32];
          tmem_ld32(t_lane + kColS + 32 * c, sv);
          uint32_t pk[16];
          if (masked)
            p_row(c, sv, true, pk);
          else
            p_row(c, sv, false, pk);
          // 16-byte chunk m of the row's 128 bytes sits at chunk m ^ (row & 7)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t off = static_cast<uint32_t>(((4 * c + m) ^ (r & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + off),
                         "r"(pk[4 * m]), "r"(pk[4 * m + 1]), "r"(pk[4 * m + 2]), "r"(pk[4 * m + 3])
                         : "memory");
          }
        }
        // phase B, dS = P (dP - D), once dP is in (the D rows came with dO_i)
        ok = mbar_wait_warp(smem_u32(&bars->dp_full), g & 1, abort, a.status);
        if (ok) ok = mbar_wait_warp(smem_u32(&bars->do_full), g & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        const float dr = sDrow[r];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dv[32];
          tmem_ld32(t_lane + kColDP + 32 * c, dv);
          uint32_t dk[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int k0 = 32 * c + 2 * t;
            dk[t] = pack_bf16x2(pf[k0] * (__uint_as_float(dv[2 * t]) - dr),
                                pf[k0 + 1] * (__uint_as_float(dv[2 * t + 1]) - dr));
          }
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t off = static_cast<uint32_t>(((4 * c + m) ^ (r & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(drow + off),
                         "r"(dk[4 * m]), "r"(dk[4 * m + 1]), "r"(dk[4 * m + 2]), "r"(dk[4 * m + 3])
                         : "memory");
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();  // P and dS are read by the tensor core next
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->pds_ready));
      }
    }
  } else {
    // ------------------------------------------ dQ^T read-out, dK / dV out
    const int wq = warp & 3;             // TMEM lane quadrant: head dims 32 wq .. 32 wq + 31 of a half
    const int rg = (warp - kDqWarp0) >> 2;  // query columns 64 rg .. 64 rg + 63; dK / dV half rg
    const uint32_t t_lane = tmem + ((static_cast<uint32_t>(wq) * 32u) << 16);
    uint32_t it = 0, g = 0;
    bool ok = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd, ++it) {
      const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
      if (item >= a.n_items) break;  // only in the last, partial round
      int bh, j;
      decode_b256(item, a, CAUSAL, bh, j);
      const int i0 = first_qblock(j, CAUSAL);
      float* const acc_bh = a.dq_acc + static_cast<size_t>(bh) * a.N * 256;
      for (int i = i0; i < a.n_qb && ok; ++i, ++g) {
        int rows = min(kTile, a.N - i * kTile);
        if (!fa_dcheck(rows <= 0 || FA_IN_RANGE(i * kTile + rows - 1, a.N), a.status))
          rows = 0;  // debug build: the rows added lie inside the head's accumulator
        for (int h = 0; h < 2; ++h) {
          const uint32_t c = 2 * g + h;
          ok = mbar_wait_warp(smem_u32(&bars->dq_full), c & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
          // lane = head dim dd, columns = this warp's 64 queries of block i;
          // TMEM is released before any reduction is issued
          uint32_t v[64];
          tmem_ld64(t_lane + kColDQ + 64 * rg, v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->dq_free));
          float* dst = acc_bh + (static_cast<size_t>(i) * kTile + 64 * rg) * 256 + 128 * h +
                       wq * 32 + lane;
#pragma unroll
          for (int q = 0; q < 64; ++q)
            if (64 * rg + q < rows) atomicAdd(dst + static_cast<size_t>(q) * 256, __uint_as_float(v[q]));
        }
      }
      if (!ok) break;
      // epilogue: dV = (dV^T)^T and dK = scale (dK^T)^T for the 64 keys,
      // head-dim half rg
      ok = mbar_wait_warp(smem_u32(&bars->acc_done), it & 1, abort, a.status);
      if (!ok) break;
      tc_fence_after();
      const int hh = bh % a.H, bb = bh / a.H;
      int keys = min(kKeys, a.N - j * kKeys);
      // debug build: the first and the last key row stored lie inside dk and dv
      if (keys > 0 &&
          !fa_dcheck(FA_IN_SPAN(a.sdv, a.BH / a.H, a.H, a.N, 256,
                                bb * a.sdv.batch + hh * a.sdv.head +
                                    static_cast<int64_t>(j * kKeys + keys - 1) * a.sdv.row, 256) &&
                         FA_IN_SPAN(a.sdk, a.BH / a.H, a.H, a.N, 256,
                                    bb * a.sdk.batch + hh * a.sdk.head +
                                        static_cast<int64_t>(j * kKeys + keys - 1) * a.sdk.row, 256),
                     a.status))
        keys = 0;
      const int dd = 128 * rg + wq * 32 + lane;
      __nv_bfloat16* dvp = a.dv + bb * a.sdv.batch + hh * a.sdv.head +
                           static_cast<int64_t>(j) * kKeys * a.sdv.row + dd;
      __nv_bfloat16* dkp = a.dk + bb * a.sdk.batch + hh * a.sdk.head +
                           static_cast<int64_t>(j) * kKeys * a.sdk.row + dd;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {  // 32 keys at a time
        uint32_t v[32], w[32];
        tmem_ld32(t_lane + kColDV + 64 * rg + 32 * cc, v);
        tmem_ld32(t_lane + kColDK + 64 * rg + 32 * cc, w);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int key = 32 * cc + t;
          if (key < keys) {
            dvp[key * a.sdv.row] = __float2bfloat16_rn(__uint_as_float(v[t]));
            dkp[key * a.sdk.row] = __float2bfloat16_rn(__uint_as_float(w[t]) * a.scale);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->acc_free));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarpB) tmem_dealloc(tmem, kTmemColsB);
}

template <bool CAUSAL>
cudaError_t launch_b256_t(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, const CUtensorMap& mdo, const Bwd256Args& a,
                          cudaStream_t stream) {
  constexpr int smem = smem_b256_bytes();
  auto kern = bwd256_dkdv_kernel<CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = min(a.n_items, p.num_sms);
  kern<<<grid, kThreadsB, smem, stream>>>(mq, mk, mv, mdo, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd256_dkdv(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mdo,
                               const Bwd256Args& a, cudaStream_t stream) {
  return p.causal ? launch_b256_t<true>(p, mq, mk, mv, mdo, a, stream)
                  : launch_b256_t<false>(p, mq, mk, mv, mdo, a, stream);
}

}  // namespace fa

// Forward at head dimension 256 ("Flash Attention v2" notes, "Detailed
// Differences", 3 "Head Dimension Support", and "Where v2 Excels Most": v2
// keeps the tiled method up to head_dim = 256).
//
// The d <= 128 kernel keeps two 128-row Q tiles per CTA with an S and an O
// accumulator each in TMEM; at d = 256 that would need 768 of the 512 TMEM
// columns. This kernel keeps ONE Q tile and double-buffers S instead:
// TMEM S0 [0,128), S1 [128,256), O [256,512). The tensor core runs
// S(j+1) while the softmax warpgroup works on S(j), then O += P(j) V(j):
//   MMA issue order  S(0) S(1) PV(0) S(2) PV(1) ... S(J-1) PV(J-2) PV(J-1).
// P(j) is written back as bf16 over the first 64 columns of S(j % 2) and
// read from TMEM by the PV MMA (A operand in TMEM).
//
// Shared memory: Q (128 x 256 bf16, 64 KiB) and a ring of five 32 KiB
// half-tiles (128 rows x 128 columns: two 64-column blocks) through which K
// and V stream, each tile as its columns 0-127 then 128-255, in the order the
// MMAs use them: K(0), K(1), V(0), K(2), V(1), ... (kv_load). PV runs as two
// N = 128 MMAs per 16-key step, one per V half.
//
// 192 threads: warps 0-3 softmax (one thread per query row = TMEM lane),
// warp 4 TMA loader, warp 5 MMA issuer. Persistent, one CTA per SM, one
// work item = (b * H + h, query tile). Every barrier wait is bounded.

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "schedule.cuh"

#ifndef FA_RESCALE_TAU_LOG2
#define FA_RESCALE_TAU_LOG2 8.0f
#endif

namespace fa {
namespace {

constexpr int kD = 256;
constexpr int kThreads256 = 192;
constexpr int kLoadWarp256 = 4;
constexpr int kMmaWarp256 = 5;
constexpr int kBlk = kTile * 64 * 2;  // 16 KiB: one 128-row x 64-column bf16 block
constexpr int kHalfBytes = 2 * kBlk;  // one half-tile: 128 rows x 128 columns
constexpr int kSlots = 5;
constexpr int kQBytes = 4 * kBlk;
constexpr uint32_t kTmemCols256 = 512;
constexpr uint32_t kColO = 256;
constexpr float kTau = FA_RESCALE_TAU_LOG2;

struct Bars256 {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kSlots], kv_empty[kSlots];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done, o_free, drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int smem256_bytes() {
  return 1024 + kQBytes + kSlots * kHalfBytes + static_cast<int>(sizeof(Bars256));
}
static_assert(smem256_bytes() <= 232448, "d = 256 forward shared memory over the limit");

struct Fwd256Args {
  __nv_bfloat16* o;
  float* lse;
  int* status;
  int N, H, BH, n_tiles, n_items;
  float scale, scale_log2;
  Strides so;
};

__device__ __forceinline__ void decode256(int item, const Fwd256Args& a, bool causal, int& bh,
                                          int& qt) {
  if (causal) {  // longest first: the last query tiles of every head come first
    qt = a.n_tiles - 1 - item / a.BH;
    bh = item % a.BH;
  } else {  // the tiles of one head adjacent, so concurrent CTAs share K/V in L2
    bh = item / a.n_tiles;
    qt = item % a.n_tiles;
  }
}

// Position of K(j) (or V(j)) among an item's half-tile loads. The MMAs use
// the tiles in the order K(0), K(1), V(0), K(2), V(1), ..., K(J - 1),
// V(J - 2), V(J - 1) (S(j + 1) is issued before PV(j)), and the loader
// issues them in that order, two half-tiles each. Loading K(j + 1) after V(j)
// instead would start K(j + 2) only once PV(j) has freed ring slots, right
// when S(j + 2) needs it: a full load latency per tile.
__device__ __forceinline__ uint32_t kv_load(bool v, int j, int J) {
  if (!v) return j == 0 ? 0u : 4u * j - 2u;
  return j == J - 1 ? 4u * J - 2u : 4u * j + 4u;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads256, 1)
    fwd256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const Fwd256Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sRing = sQ + kQBytes;
  Bars256* bars = reinterpret_cast<Bars256*>(smem + kQBytes + kSlots * kHalfBytes);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_empty), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->s_full[t]), 1);
      mbar_init(smem_u32(&bars->p_full[t]), 4);  // one elected lane per softmax warp
    }
    mbar_init(smem_u32(&bars->o_done), 1);
    mbar_init(smem_u32(&bars->o_free), 4);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp256) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols256);
    tmem_relinquish();
  }
  if (warp == kLoadWarp256 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kLoadWarp256) {
    // ---------------------------------------------------------------- loader
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t it = 0, n = 0;  // items loaded, half-tiles loaded
      bool ok = true;
      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd, ++it) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= a.n_items) break;  // only in the last, partial round
        int bh, qt;
        decode256(item, a, CAUSAL, bh, qt);
        const int hh = bh % a.H, bb = bh / a.H;
        const int J = CAUSAL ? qt + 1 : a.n_tiles;
        ok = mbar_wait(smem_u32(&bars->q_empty), (it & 1) ^ 1, abort, a.status);
        if (!ok) break;
        {
          const uint32_t bar = smem_u32(&bars->q_full);
          mbar_arrive_expect_tx(bar, kQBytes);
          tma_load_5d(sQ, &tmQ, bar, 0, qt * kTile, 0, hh, bb, pol_q);  // all four column blocks
        }
        // tiles in the order the MMAs consume them: K(0), then K(j), V(j - 1)
        // for j = 1 .. J - 1, then V(J - 1) (see kv_load)
        for (int t = 0; t < 2 * J && ok; ++t) {
          const bool is_v = t > 0 && (t == 2 * J - 1 || (t & 1) == 0);
          const int tile = is_v ? (t == 2 * J - 1 ? J - 1 : t / 2 - 1) : (t + 1) / 2;
          for (int w = 0; w < 2; ++w, ++n) {  // columns 0-127, then 128-255
            const uint32_t s = n % kSlots;
            ok = mbar_wait(smem_u32(&bars->kv_empty[s]), ((n / kSlots) & 1) ^ 1, abort,
                           a.status);
            if (!ok) break;
            const uint32_t bar = smem_u32(&bars->kv_full[s]);
            const CUtensorMap* map = is_v ? &tmV : &tmK;
            mbar_arrive_expect_tx(bar, kHalfBytes);  // column blocks 2w, 2w + 1 in one copy
            tma_load_5d(sRing + s * kHalfBytes, map, bar, 0, tile * kTile, 2 * w, hh, bb, pol_kv);
          }
        }
      }
      // producer tail: every stage released before the CTA exits (after an
      // abort, the copies already issued are allowed to land)
      const uint32_t m = min(n, static_cast<uint32_t>(kSlots));
      for (uint32_t u = n - m; u < n; ++u) {
        const uint32_t s = u % kSlots, ph = (u / kSlots) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->kv_empty[s]), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->kv_full[s]), ph, 100000000ull);
      }
      if (it > 0) {
        const uint32_t ph = (it - 1) & 1;
        if (ok) ok = mbar_wait(smem_u32(&bars->q_empty), ph, abort, a.status);
        if (!ok) mbar_drain(smem_u32(&bars->q_full), ph, 100000000ull);
      }
    }
  } else if (warp == kMmaWarp256) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kTile, 128, false, true);
      uint32_t it = 0, n = 0, g0 = 0;
      bool ok = true;
      // S(g) = Q K^T into S(g % 2), over 16 steps of 16 head-dim columns; the
      // K half-tiles come from the ring, the Q blocks from the Q region
      auto issue_s = [&](uint32_t g, uint32_t kslot0, uint32_t kslot1) {
        const uint32_t dst = tmem + 128u * (g & 1u);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint32_t kslot = kk < 8 ? kslot0 : kslot1;
          const uint32_t k_off = ((kk >> 2) & 1) * kBlk + (kk & 3) * 32;
          const SmemDesc da = make_desc_sw128(opaque_u32(sQ + (kk >> 2) * kBlk + (kk & 3) * 32), 16, 1024);
          const SmemDesc db = make_desc_sw128(opaque_u32(sRing + kslot * kHalfBytes + k_off), 16, 1024);
          mma_ss(dst, desc_at(da, 0), desc_at(db, 0), idesc_s, kk > 0);
        }
      };
      // O[:, 128 h .. 128 h + 127] (+)= P(g) V[:, 128 h ..] for one V half
      auto issue_pv = [&](uint32_t g, int h, uint32_t vslot, bool accumulate) {
        const uint32_t dst = tmem + kColO + 128u * h;
        const uint32_t pa = tmem + 128u * (g & 1u);
        const SmemDesc db = make_desc_sw128(opaque_u32(sRing + vslot * kHalfBytes), kBlk, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(dst, pa + kk * 8, desc_at(db, kk * 2048), idesc_o,
                 (accumulate || kk > 0) ? 1u : 0u);
      };
      for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd, ++it) {
        const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
        if (item >= a.n_items) break;  // only in the last, partial round
        int bh, qt;
        decode256(item, a, CAUSAL, bh, qt);
        const int J = CAUSAL ? qt + 1 : a.n_tiles;
        ok = mbar_wait(smem_u32(&bars->q_full), it & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; j <= J && ok; ++j) {
          if (j < J) {  // S(j)
            const uint32_t nk0 = n + kv_load(false, j, J), nk1 = nk0 + 1;
            const uint32_t s0 = nk0 % kSlots, s1 = nk1 % kSlots;
            ok = mbar_wait(smem_u32(&bars->kv_full[s0]), (nk0 / kSlots) & 1, abort, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bars->kv_full[s1]), (nk1 / kSlots) & 1, abort, a.status);
            if (!ok) break;
            tc_fence_after();
            issue_s(g0 + j, s0, s1);
            mma_commit(smem_u32(&bars->s_full[(g0 + j) & 1]));
            mma_commit(smem_u32(&bars->kv_empty[s0]));
            mma_commit(smem_u32(&bars->kv_empty[s1]));
            if (j == J - 1) mma_commit(smem_u32(&bars->q_empty));
          }
          if (j >= 1) {  // PV(j - 1)
            const uint32_t g = g0 + j - 1;
            if (j == 1 && it > 0) {  // the previous item's epilogue has read O
              ok = mbar_wait(smem_u32(&bars->o_free), (it - 1) & 1, abort, a.status);
              if (!ok) break;
            }
            ok = mbar_wait(smem_u32(&bars->p_full[g & 1]), (g >> 1) & 1, abort, a.status);
            if (!ok) break;
            const uint32_t nv0 = n + kv_load(true, j - 1, J), nv1 = nv0 + 1;
            const uint32_t s0 = nv0 % kSlots, s1 = nv1 % kSlots;
            ok = mbar_wait(smem_u32(&bars->kv_full[s0]), (nv0 / kSlots) & 1, abort, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bars->kv_full[s1]), (nv1 / kSlots) & 1, abort, a.status);
            if (!ok) break;
            tc_fence_after();
            issue_pv(g, 0, s0, j > 1);
            issue_pv(g, 1, s1, j > 1);
            mma_commit(smem_u32(&bars->o_done));
            mma_commit(smem_u32(&bars->kv_empty[s0]));
            mma_commit(smem_u32(&bars->kv_empty[s1]));
          }
        }
        n += 4 * J;
        g0 += J;
      }
      mma_commit(smem_u32(&bars->drain));
      mbar_drain(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = warp * 32 + lane;  // query row within the tile = TMEM lane
    const uint32_t t_lane = tmem + ((static_cast<uint32_t>(warp) * 32u) << 16);
    const uint32_t tO = t_lane + kColO;
    const float sl2 = a.scale_log2;
    const float NEG_INF = __int_as_float(0xff800000);
    uint32_t g0 = 0;
    bool ok = true;
    for (int rnd = 0; rnd * static_cast<int>(gridDim.x) < a.n_items && ok; ++rnd) {
      const int item = sched_item(rnd, blockIdx.x, gridDim.x, CAUSAL);
      if (item >= a.n_items) break;  // only in the last, partial round
      int bh, qt;
      decode256(item, a, CAUSAL, bh, qt);
      const int J = CAUSAL ? qt + 1 : a.n_tiles;
      float m = NEG_INF, l = 0.f;
      for (int j = 0; j < J; ++j) {
        const uint32_t g = g0 + j;
        const uint32_t tS = t_lane + 128u * (g & 1u);
        ok = mbar_wait_warp(smem_u32(&bars->s_full[g & 1]), (g >> 1) & 1, abort, a.status);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128(tS, sr);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        // masks: causal diagonal tile, and keys past N in the last tile
        int lim = 127;
        if (CAUSAL && j == qt) lim = r;
        if (j == a.n_tiles - 1) lim = min(lim, a.N - 1 - j * kTile);
        const bool masked = lim < 127;
        if (masked) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c > lim) ? NEG_INF : s[c];
        }
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
        } else if ((mt - m) * sl2 > kTau) {
          m_use = mt;
          alpha = ex2_approx((m - mt) * sl2);
          grow = true;
        }
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
          float p0 = ex2_approx(x.x);
          float p1 = ex2_approx(x.y);
          acc[c & 3] = fadd2(acc[c & 3], make_float2(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
        const float2 a03 = fadd2(a01, a23);
        l = alpha * l + (a03.x + a03.y);
        tmem_st64(tS, pk);
        if (__any_sync(0xffffffffu, grow)) {
          // O holds the sum up to tile j - 1 once PV(g - 1) has completed;
          // S(g) complete implies PV(g - 2) complete, so o_done is at phase
          // g - 1 or past it and the parity wait is exact
          ok = mbar_wait_warp(smem_u32(&bars->o_done), (g - 1) & 1, abort, a.status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < kD / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
            tmem_st32(tO + cc * 32, o);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[g & 1]));
        m = m_use;
      }
      if (!ok) break;
      // epilogue: O / l in bf16 and the log-sum-exp, then O is free. S(g)
      // is issued before PV(g - 1), so here PV(g_last - 1) may still be
      // pending and o_done a whole phase behind: wait for it first, or the
      // parity wait for PV(g_last) would see that older phase as done. (S(g)
      // complete implies PV(g - 2) complete, so it lags by one at most.)
      const uint32_t g_last = g0 + J - 1;
      if (g_last > 0) {
        ok = mbar_wait_warp(smem_u32(&bars->o_done), (g_last - 1) & 1, abort, a.status);
        if (!ok) break;
      }
      ok = mbar_wait_warp(smem_u32(&bars->o_done), g_last & 1, abort, a.status);
      if (!ok) break;
      tc_fence_after();
      const int row = qt * kTile + r;
      bool store = row < a.N;
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = a.o + (bh / a.H) * a.so.batch + (bh % a.H) * a.so.head +
                            static_cast<int64_t>(row) * a.so.row;
#ifdef FA_DEBUG
      if (store) store = fa_dcheck(in_span(a.so, a.BH / a.H, a.H, a.N, kD, orow - a.o, kD), a.status);
#endif
#pragma unroll 1
      for (int cc = 0; cc < kD / 32; ++cc) {
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
      if (store)
        a.lse[static_cast<size_t>(bh) * a.N + row] =
            fmaf(m, a.scale, lg2_approx(l) * 0.69314718055994531f);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->o_free));
      g0 += J;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp256) tmem_dealloc(tmem, kTmemCols256);
}

template <bool CAUSAL>
cudaError_t launch256_t(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                        const CUtensorMap& mv, const Fwd256Args& a, cudaStream_t stream) {
  constexpr int smem = smem256_bytes();
  auto kern = fwd256_kernel<CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = min(a.n_items, p.num_sms);
  kern<<<grid, kThreads256, smem, stream>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd256(const Problem& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  // 5-D maps: Q's copy spans all four 64-column blocks, a K or V half-tile's two
  if (!make_tile_map(&mq, q, p.B, p.H, p.N, p.d, p.st[kQ], kTile, 4) ||
      !make_tile_map(&mk, k, p.B, p.H, p.N, p.d, p.st[kK], kTile, 2) ||
      !make_tile_map(&mv, v, p.B, p.H, p.N, p.d, p.st[kV], kTile, 2))
    return cudaErrorInvalidValue;
  Fwd256Args a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = p.status;
  a.N = p.N;
  a.H = p.H;
  a.BH = p.B * p.H;
  a.n_tiles = (p.N + kTile - 1) / kTile;
  a.n_items = a.BH * a.n_tiles;
  a.scale = p.scale;
  a.scale_log2 = clamped_scale_log2(p.scale);
  a.so = p.st[kO];
  return p.causal ? launch256_t<true>(p, mq, mk, mv, a, stream)
                  : launch256_t<false>(p, mq, mk, mv, a, stream);
}

}  // namespace fa

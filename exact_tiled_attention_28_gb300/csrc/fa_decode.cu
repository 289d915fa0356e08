// Decode: a few new query rows per (batch, head) against a long key/value
// cache, split along the keys.
//
// The pages name serving as a use of the method ("flashattention-2"
// glossary, "Adoption": vLLM's attention backend; "Flash Attention v2" notes,
// "Performance Comparison: v1 vs v2": 256-token generation, continuous
// batching). With Nq <= 16 rows per head the work is reading K and V once:
// 4 Nq flops per 4 bytes of cache, far left of the tensor-core ridge, so these
// kernels use the CUDA cores and are built around HBM bandwidth.
//
// The exact result is kept by splitting the keys of each (batch, head) into
// contiguous ranges, one per CTA; each range yields its own softmax
// statistics and normalised output, and the ranges are merged by their
// log-sum-exp, the same identity the tiled online softmax rests on ("Flash
// Attention v2" notes, "Detailed Algorithm Comparison", forward pass: the
// running max m, the running sum l and the rescale factor exp(m - m_new)).
//
// decode_split_kernel<D, NQ>: grid (B*H, splits), 160 threads.
//   warp 4 (one lane) streams 128-key K and V tiles of the split through a
//   ring of shared-memory stages with TMA;
//   warps 0-3 each own 32 keys of every tile: lane = key for S = q . k
//   (K rows read 16 bytes at a time; the 128-byte swizzle of the tile spreads
//   the 32 rows over all banks), a per-warp online softmax, and lanes over
//   the head dimension for O += p v (p broadcast by shuffles);
//   at the end the four warps merge in shared memory and the CTA writes
//   either the final O and LSE (one split) or its split's normalised O and
//   log2-domain LSE to the workspace.
// decode_combine_kernel<D>: one warp per (batch, head, row) merges the splits.
//
// Scores are kept in log2 units (q is pre-multiplied by scale * log2 e), so
// exponentials are exp2. The causal mask is aligned at the bottom right:
// row r of Nq sees key j when j <= r + nk - Nq.

#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecConsumerWarps = 4;
constexpr int kDecThreads = 32 * (kDecConsumerWarps + 1);
constexpr int kDecProducerWarp = kDecConsumerWarps;
constexpr int kDecBlockBytes = kTile * 64 * 2;  // one 128-row x 64-column bf16 block

template <int D>
struct DecCfg {
  static constexpr int kColBlocks = (D + 63) / 64;
  static constexpr int kTileBytes = kColBlocks * kDecBlockBytes;  // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = D > 64 ? 3 : 6;
  static constexpr int kE = D / 32;  // head-dim elements per lane in O
};

struct DecBars {
  uint64_t full[6], empty[6];
  int abort;
};

template <int D, int NQ>
constexpr int dec_smem_bytes() {
  // stages, then q (fp32) and the barriers; the warps' merge reuses the stages
  return 1024 + DecCfg<D>::kStages * DecCfg<D>::kStageBytes + NQ * D * 4 +
         static_cast<int>(sizeof(DecBars));
}
static_assert(dec_smem_bytes<128, 16>() <= 232448, "decode shared memory over the limit");
static_assert(DecCfg<128>::kStages * DecCfg<128>::kStageBytes >=
                  kDecConsumerWarps * 16 * (128 + 2) * 4,
              "merge area does not fit in the stages");

struct DecodeArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;       // [B, H, Nq], natural log
  float* part_o;    // [B*H, splits, NQ, D]: each split's normalised O
  float* part_lse;  // [B*H, splits, NQ]: each split's LSE in log2 units
  const int* cache_seqlens;
  int* status;
  int H, Nq, Nk, splits, tiles_per_split, causal;
  float scale_log2;
  Strides sq, so;
  int B;  // debug build: index checks
};

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t ld_shared_b32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint16_t ld_shared_b16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// q is re-read from shared memory for every tile: volatile loads keep the
// compiler from hoisting NQ x D values out of the tile loop into registers.
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Byte offset of element (row, col) in a 128B-swizzled tile of 64-column blocks.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return static_cast<uint32_t>((col >> 6) * kDecBlockBytes + row * 128 +
                               ((((col >> 3) & 7) ^ (row & 7)) << 4) + (col & 7) * 2);
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D, int NQ>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
  using Cfg = DecCfg<D>;
  constexpr int S = Cfg::kStages;
  constexpr int E = Cfg::kE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sStage = smem_u32(smem);
  float* qf = reinterpret_cast<float*>(smem + S * Cfg::kStageBytes);  // [NQ][D]
  const uint32_t sQf = smem_u32(qf);
  DecBars* bars = reinterpret_cast<DecBars*>(smem + S * Cfg::kStageBytes + NQ * D * 4);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int split = blockIdx.y;
  const int b = bh / a.H, h = bh - b * a.H;
  int nk = a.Nk;
  if (a.cache_seqlens != nullptr) {
    const int v = __ldg(a.cache_seqlens + b);
    nk = min(max(v, 0), a.Nk);
    if (threadIdx.x == 0 && split == 0 && h == 0 && (v < 0 || v > a.Nk))
      atomicCAS(a.status, DEV_OK, DEV_BADARG);
  }
  const int n_tiles = (nk + kTile - 1) / kTile;
  const int t0 = split * a.tiles_per_split;
  const int nt = max(min(t0 + a.tiles_per_split, n_tiles) - t0, 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), kDecConsumerWarps);
    }
    bars->abort = 0;
    fence_barrier_init();
  }
  // q of this (batch, head), times scale * log2 e; rows past Nq are zero
  for (int i = threadIdx.x; i < NQ * D; i += kDecThreads) {
    const int r = i / D, c = i - (i / D) * D;
    float x = 0.f;
    if (r < a.Nq)
      x = __bfloat162float(a.q[b * a.sq.batch + h * a.sq.head + static_cast<int64_t>(r) * a.sq.row + c]) *
          a.scale_log2;
    qf[i] = x;
  }
  __syncthreads();

  if (warp == kDecProducerWarp) {
    // ------------------------------------------------------------- producer
    if (lane == 0 && nt > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t pol = policy_evict_first();  // the cache is read once
      bool ok = true;
      int i = 0;
      for (; i < nt && ok; ++i) {
        const int s = i % S;
        ok = mbar_wait(smem_u32(&bars->empty[s]), ((i / S) & 1) ^ 1, abort, a.status);
        if (!ok) break;
        const uint32_t bar = smem_u32(&bars->full[s]);
        const uint32_t st = sStage + s * Cfg::kStageBytes;
        mbar_arrive_expect_tx(bar, Cfg::kStageBytes);
        for (int cb = 0; cb < Cfg::kColBlocks; ++cb) {
          tma_load_4d(st + cb * kDecBlockBytes, &tmK, bar, 64 * cb, (t0 + i) * kTile, h, b, pol);
          tma_load_4d(st + Cfg::kTileBytes + cb * kDecBlockBytes, &tmV, bar, 64 * cb,
                      (t0 + i) * kTile, h, b, pol);
        }
      }
      if (!ok) {  // after an abort, let the copies in flight land before the CTA exits
        for (int u = max(i - S, 0); u < i; ++u)
          mbar_drain(smem_u32(&bars->full[u % S]), (u / S) & 1, 100000000ull);
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  const float NEG_INF = __int_as_float(0xff800000);
  float m[NQ], lsum[NQ], acc[NQ][E];
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    m[r] = NEG_INF;
    lsum[r] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
  }
  const int kl = warp * 32 + lane;  // key of this lane within a tile
  bool ok = true;
  for (int i = 0; i < nt; ++i) {
    const int s = i % S;
    ok = mbar_wait_warp(smem_u32(&bars->full[s]), (i / S) & 1, abort, a.status);
    if (!ok) break;
    const uint32_t Kt = sStage + s * Cfg::kStageBytes;
    const uint32_t Vt = Kt + Cfg::kTileBytes;
    // S row entries for this lane's key, all query rows
    float sc[NQ];
#pragma unroll
    for (int r = 0; r < NQ; ++r) sc[r] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 kv = ld_shared_v4(Kt + swz(kl, 8 * c));
      const float k[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                          bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        const float4 qa = ld_shared_f4(sQf + (r * D + 8 * c) * 4);
        const float4 qb = ld_shared_f4(sQf + (r * D + 8 * c + 4) * 4);
        float x = sc[r];
        x = fmaf(qa.x, k[0], x);
        x = fmaf(qa.y, k[1], x);
        x = fmaf(qa.z, k[2], x);
        x = fmaf(qa.w, k[3], x);
        x = fmaf(qb.x, k[4], x);
        x = fmaf(qb.y, k[5], x);
        x = fmaf(qb.z, k[6], x);
        x = fmaf(qb.w, k[7], x);
        sc[r] = x;
      }
    }
    // masks and the per-warp online softmax of this tile
    const int key = (t0 + i) * kTile + kl;
    float p[NQ];
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      const bool vis = key < nk && (!a.causal || key <= r + nk - a.Nq);
      const float x = vis ? sc[r] : NEG_INF;
      const float m_new = fmaxf(m[r], warp_max(x));
      const float m_use = m_new == NEG_INF ? 0.f : m_new;
      const float alpha = ex2_approx(m[r] - m_use);
      p[r] = ex2_approx(x - m_use);
      lsum[r] = fmaf(lsum[r], alpha, p[r]);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[r][e] *= alpha;
      m[r] = m_new;
    }
    // O += p V over the warp's 32 keys; lane owns head-dim elements lane*E ..
#pragma unroll 4
    for (int kk = 0; kk < 32; ++kk) {
      const int vr = warp * 32 + kk;
      float v[E];
      if constexpr (E == 4) {
        const uint2 w = ld_shared_v2(Vt + swz(vr, 4 * lane));
        v[0] = bf16_lo(w.x);
        v[1] = bf16_hi(w.x);
        v[2] = bf16_lo(w.y);
        v[3] = bf16_hi(w.y);
      } else if constexpr (E == 2) {
        const uint32_t w = ld_shared_b32(Vt + swz(vr, 2 * lane));
        v[0] = bf16_lo(w);
        v[1] = bf16_hi(w);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
          v[e] = __uint_as_float(static_cast<uint32_t>(ld_shared_b16(Vt + swz(vr, E * lane + e))) << 16);
      }
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        const float pr = __shfl_sync(0xffffffffu, p[r], kk);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[r][e] = fmaf(pr, v[e], acc[r][e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars->empty[s]));
  }

  // merge the four warps (the stages are free: every tile was consumed)
  named_bar_sync(1, kDecConsumerWarps * 32);
  float* wm = reinterpret_cast<float*>(smem);       // [4][NQ]
  float* wl = wm + kDecConsumerWarps * NQ;          // [4][NQ]
  float* wo = wl + kDecConsumerWarps * NQ;          // [4][NQ][D]
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    const float lw = warp_sum(lsum[r]);
    if (lane == 0) {
      wm[warp * NQ + r] = m[r];
      wl[warp * NQ + r] = lw;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) wo[(warp * NQ + r) * D + E * lane + e] = acc[r][e];
  }
  named_bar_sync(1, kDecConsumerWarps * 32);
  const bool direct = a.splits == 1;
  for (int idx = threadIdx.x; idx < NQ * D; idx += kDecConsumerWarps * 32) {
    const int r = idx / D, c = idx - (idx / D) * D;
    float M = NEG_INF;
#pragma unroll
    for (int w = 0; w < kDecConsumerWarps; ++w) M = fmaxf(M, wm[w * NQ + r]);
    float L = 0.f, O = 0.f;
    if (M != NEG_INF) {
#pragma unroll
      for (int w = 0; w < kDecConsumerWarps; ++w) {
        const float f = ex2_approx(wm[w * NQ + r] - M);
        L = fmaf(wl[w * NQ + r], f, L);
        O = fmaf(wo[(w * NQ + r) * D + c], f, O);
      }
    }
    const float out = L > 0.f ? O / L : 0.f;
    const float lse2 = L > 0.f ? M + lg2_approx(L) : NEG_INF;
    if (direct) {
      const int64_t off = b * a.so.batch + h * a.so.head + static_cast<int64_t>(r) * a.so.row + c;
      if (r < a.Nq && fa_dcheck(FA_IN_SPAN(a.so, a.B, a.H, a.Nq, D, off, 1), a.status)) {
        a.o[off] = __float2bfloat16_rn(out);
        if (c == 0)
          a.lse[static_cast<size_t>(bh) * a.Nq + r] =
              lse2 == NEG_INF ? NEG_INF : lse2 * 0.69314718055994531f;
      }
    } else {
      const size_t part = (static_cast<size_t>(bh) * a.splits + split) * NQ + r;
      a.part_o[part * D + c] = out;
      if (c == 0) a.part_lse[part] = lse2;
    }
  }
}

// One warp per (batch, head, row): O = sum_s 2^(lse_s - lse) O_s with
// 2^lse = sum_s 2^lse_s (log2 units); splits without a visible key carry
// lse_s = -inf and weigh nothing.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeArgs a, int nq_pad,
                                                             int rows) {
  const int gw = static_cast<int>((static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= rows) return;
  const int bh = gw / a.Nq, r = gw - (gw / a.Nq) * a.Nq;
  const int b = bh / a.H, h = bh - b * a.H;
  const float NEG_INF = __int_as_float(0xff800000);
  const size_t base = static_cast<size_t>(bh) * a.splits * nq_pad + r;
  float M = NEG_INF;
  for (int s = lane; s < a.splits; s += 32) M = fmaxf(M, a.part_lse[base + static_cast<size_t>(s) * nq_pad]);
  M = warp_max(M);
  float L = 0.f;
  if (M != NEG_INF)
    for (int s = lane; s < a.splits; s += 32)
      L += ex2_approx(a.part_lse[base + static_cast<size_t>(s) * nq_pad] - M);
  L = warp_sum(L);
  const int64_t roff = b * a.so.batch + h * a.so.head + static_cast<int64_t>(r) * a.so.row;
  if (!fa_dcheck(FA_IN_SPAN(a.so, a.B, a.H, a.Nq, D, roff, D), a.status)) return;
  __nv_bfloat16* orow = a.o + roff;
  for (int c = lane; c < D; c += 32) {
    float O = 0.f;
    if (M != NEG_INF) {
      for (int s = 0; s < a.splits; ++s) {
        const size_t part = base + static_cast<size_t>(s) * nq_pad;
        const float f = ex2_approx(a.part_lse[part] - M);
        O = fmaf(a.part_o[part * D + c], f, O);
      }
    }
    orow[c] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
  }
  if (lane == 0)
    a.lse[static_cast<size_t>(bh) * a.Nq + r] =
        L > 0.f ? (M + lg2_approx(L)) * 0.69314718055994531f : NEG_INF;
}


template <int D, int NQ>
cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                            int BH, cudaStream_t stream) {
  constexpr int smem = dec_smem_bytes<D, NQ>();
  auto kern = decode_split_kernel<D, NQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(BH, a.splits), kDecThreads, smem, stream>>>(mk, mv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  const int rows = BH * a.Nq;
  const int blocks = (rows + 7) / 8;  // 8 warps per block
  decode_combine_kernel<D><<<blocks, 256, 0, stream>>>(a, NQ, rows);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                            int BH, cudaStream_t stream) {
  switch (nq_pad_of(a.Nq)) {
    case 1: return launch_decode_t<D, 1>(a, mk, mv, BH, stream);
    case 2: return launch_decode_t<D, 2>(a, mk, mv, BH, stream);
    case 4: return launch_decode_t<D, 4>(a, mk, mv, BH, stream);
    case 8: return launch_decode_t<D, 8>(a, mk, mv, BH, stream);
    default: return launch_decode_t<D, 16>(a, mk, mv, BH, stream);
  }
}

}  // namespace

int nq_pad_of(int Nq) {
  int n = 1;
  while (n < Nq) n *= 2;
  return n;
}

cudaError_t launch_decode_combine(const Problem& p, const float* part_o, const float* part_lse,
                                  int splits, void* o, float* lse, cudaStream_t stream) {
  DecodeArgs a{};
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.part_o = const_cast<float*>(part_o);
  a.part_lse = const_cast<float*>(part_lse);
  a.status = p.status;
  a.H = p.H;
  a.B = p.B;
  a.Nq = p.N;
  a.splits = splits;
  a.so = p.st[kO];
  const int rows = p.B * p.H * p.N;
  const int blocks = (rows + 7) / 8;  // 8 warps per block
  const int nq_pad = nq_pad_of(p.N);
  switch (p.d) {
    case 32: decode_combine_kernel<32><<<blocks, 256, 0, stream>>>(a, nq_pad, rows); break;
    case 64: decode_combine_kernel<64><<<blocks, 256, 0, stream>>>(a, nq_pad, rows); break;
    case 96: decode_combine_kernel<96><<<blocks, 256, 0, stream>>>(a, nq_pad, rows); break;
    default: decode_combine_kernel<128><<<blocks, 256, 0, stream>>>(a, nq_pad, rows); break;
  }
  return cudaGetLastError();
}

// Splits per (batch, head): as many as fit one wave of one CTA per SM (the
// stages take most of the shared memory), at least one tile per split. On
// GB300 this beat plans that fill several whole waves (93K valid keys of a
// 128K cache, B = 1, H = 32: 6.1 against 5.7 TB/s): a CTA's pipeline fill is
// paid again at every wave, and splits planned on the cache size idle where
// the valid keys end.
DecodePlan decode_plan(int B, int H, int Nk, int num_sms) {
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int tiles = (Nk + kTile - 1) / kTile;
  int splits = bh >= num_sms ? 1 : static_cast<int>(std::min<int64_t>(tiles, num_sms / bh));
  splits = std::max(std::min(splits, kDecodeMaxSplits), 1);
  const int tps = (tiles + splits - 1) / splits;
  return DecodePlan{(tiles + tps - 1) / tps, tps};
}

int decode_tc_splits(int B, int H, int Nk, int num_sms) {
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int tiles = (Nk + kTile - 1) / kTile;
  if (bh >= num_sms) return 1;
  const int lo = static_cast<int>((num_sms + bh - 1) / bh);
  const int hi = std::max(std::min(tiles, kDecodeMaxSplits), 1);
  int best = std::min(lo, hi);
  double best_fill = 0.0;
  for (int s = std::min(lo, hi); s <= hi; ++s) {
    const int64_t items = bh * s;
    const int64_t rounds = (items + num_sms - 1) / num_sms;
    const double fill = static_cast<double>(items) / static_cast<double>(rounds * num_sms);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = s;
    }
    if (fill >= 0.95) break;
  }
  return best;
}

size_t decode_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_sms) {
  const DecodePlan pl = decode_plan(B, H, Nk, num_sms);
  int splits = pl.splits == 1 ? 0 : pl.splits;
  // Nq >= 8 at d = 64 and 128 runs the tensor-core forward with its own split count
  if (Nq >= kDecodeTensorMinQ && fwd_split_supported(d) && static_cast<int64_t>(B) * H < num_sms)
    splits = std::max(splits, decode_tc_splits(B, H, Nk, num_sms));
  if (splits <= 1) return 0;
  return static_cast<size_t>(B) * H * splits * nq_pad_of(Nq) * (d + 1) * 4;
}

cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, const int* cache_seqlens, void* workspace,
                          cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!make_tile_map(&mk, k, p.B, p.H, p.Nk, p.d, p.st[kK]) ||
      !make_tile_map(&mv, v, p.B, p.H, p.Nk, p.d, p.st[kV]))
    return cudaErrorInvalidValue;
  const DecodePlan pl = decode_plan(p.B, p.H, p.Nk, p.num_sms);
  const int BH = p.B * p.H;
  DecodeArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  float* ws = static_cast<float*>(workspace);
  const size_t parts = static_cast<size_t>(BH) * pl.splits * nq_pad_of(p.N);
  a.part_o = ws;
  a.part_lse = ws == nullptr ? nullptr : ws + parts * p.d;
  a.cache_seqlens = cache_seqlens;
  a.status = p.status;
  a.H = p.H;
  a.B = p.B;
  a.Nq = p.N;
  a.Nk = p.Nk;
  a.splits = pl.splits;
  a.tiles_per_split = pl.tiles_per_split;
  a.causal = p.causal;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.sq = p.st[kQ];
  a.so = p.st[kO];
  switch (p.d) {
    case 32: return launch_decode_d<32>(a, mk, mv, BH, stream);
    case 64: return launch_decode_d<64>(a, mk, mv, BH, stream);
    case 96: return launch_decode_d<96>(a, mk, mv, BH, stream);
    default: return launch_decode_d<128>(a, mk, mv, BH, stream);
  }
}

}  // namespace fa

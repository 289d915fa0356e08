// Geometry of one (sequence, head) in a batch of sequences with unequal
// query and key lengths, shared by the forward and backward kernels.
//
// The pages state the method for one length N; for batches of requests of
// different lengths ("Flash Attention v2" notes, "Performance Comparison: v1
// vs v2", continuous batching) they fix no convention. Here Nq query rows
// attend to Nk keys with the causal mask aligned at the bottom right: query i
// sees key j when j <= i + Nk - Nq.
#pragma once

#include "kernels.h"

namespace fa {

// What every kernel of a batch with unequal lengths needs to place a
// sequence. Dense batch (cu_q null): sequence b is batch coordinate b with
// Nq query and Nk key rows. Packed batch: sequence b owns rows
// cu_q[b]..cu_q[b+1]-1 of q (and o, dO, dq) and cu_k[b]..cu_k[b+1]-1 of k
// and v, at batch coordinate 0; the buffers hold rows_q and rows_k rows per
// head, and no length exceeds max_q / max_k.
struct VarGeom {
  const int* cu_q;
  const int* cu_k;
  int H, Nq, Nk, rows_q, rows_k, max_q, max_k;
};

struct Seq {
  int bb, hh;  // batch and head coordinates in the tensors
  int q0, k0;  // first query row and first key row
  int nq, nk;  // query rows and key rows
  int pst;     // first row of the sequence in the backward's padded D / lse2 rows
};

// Sequence-and-head index sh = b * H + h. Packed offsets are clamped to the
// buffers, so that malformed offsets give wrong results but every row index
// stays inside the tensors (a separate check reports them). KLENS: a dense
// batch whose cu_k holds B per-sequence key counts (a key/value cache with
// valid lengths), clamped to 0..Nk.
template <bool KLENS = false>
__device__ __forceinline__ Seq seq_of(int sh, const VarGeom& g) {
  Seq s;
  const int b = sh / g.H;
  s.hh = sh - b * g.H;
  if (g.cu_q != nullptr) {
    const int q0 = min(max(__ldg(g.cu_q + b), 0), g.rows_q);
    const int q1 = min(max(__ldg(g.cu_q + b + 1), q0), g.rows_q);
    const int k0 = min(max(__ldg(g.cu_k + b), 0), g.rows_k);
    const int k1 = min(max(__ldg(g.cu_k + b + 1), k0), g.rows_k);
    s.bb = 0;
    s.q0 = q0;
    s.nq = min(q1 - q0, g.max_q);
    s.k0 = k0;
    s.nk = min(k1 - k0, g.max_k);
    // sequences start on a 128-row boundary of the padded rows, with one
    // spare tile per sequence: roundup(q0, 128) + 128 b
    s.pst = ((q0 + kTile - 1) / kTile + b) * kTile;
  } else {
    s.bb = b;
    s.q0 = 0;
    s.k0 = 0;
    s.nq = g.Nq;
    s.nk = KLENS ? min(max(__ldg(g.cu_k + b), 0), g.Nk) : g.Nk;
    s.pst = 0;
  }
  return s;
}

// One warp turns counts in a[1..n] into their running sums; a[0] = 0.
__device__ __forceinline__ void scan_counts_warp(int* a, int n, int lane) {
  const int per = (n + 31) / 32;
  const int lo = 1 + lane * per, hi = min(lo + per, n + 1);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += a[i];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - sum;  // exclusive prefix of this lane's chunk
  for (int i = lo; i < hi; ++i) {
    run += a[i];
    a[i] = run;
  }
  if (lane == 0) a[0] = 0;
}

// A compacted, longest-first schedule of a packed batch, so that no work
// item of the persistent grid lies past its sequence. Sequence b owns c_b
// "levels" (query-tile pairs in the forward, key tiles in the backward),
// each of H items. Sequences are sorted by c_b, largest first, and by index
// among equal c_b (sorted[]): a stable order, so that every block that builds
// the schedule gets the same one.
//  - non-causal (every level of a sequence costs the same): sequence by
//    sequence in sorted order, the levels of a head adjacent; pre[r] = items
//    of the sorted sequences before rank r.
//  - causal (the cost grows with the level; larger first): level by level,
//    every (sequence, head) that has the level in sorted order; start[t] =
//    items before the t-th level visited, kcount[v] = sequences with more
//    than v levels (= the rank where the sequences with v levels start).
// The layout of the arrays is [hist P+1][kcount P+1][start P+1][sorted n]
// [pre n+1] ints, P = the largest c_b (the caller sizes the region).
struct Sched {
  int* hist;
  int* kcount;
  int* start;
  int* sorted;
  int* pre;
};

__device__ __forceinline__ Sched sched_arrays(int* base, int n, int P) {
  Sched s;
  s.hist = base;
  s.kcount = s.hist + (P + 1);
  s.start = s.kcount + (P + 1);
  s.sorted = s.start + (P + 1);
  s.pre = s.sorted + n;
  return s;
}

__host__ __device__ constexpr size_t sched_ints(int n, int P) {
  return 3 * (static_cast<size_t>(P) + 1) + 2 * static_cast<size_t>(n) + 1;
}

// A one-block builder of kSchedBuildThreads threads places with every warp
// when given this much scratch.
constexpr int kSchedBuildThreads = 1024;
__host__ __device__ constexpr size_t sched_build_scratch_ints(int P) {
  return static_cast<size_t>(kSchedBuildThreads / 32) * (static_cast<size_t>(P) + 1);
}

// Builds the schedule with the threads of one block; count(b) gives c_b
// (clamped to P); the total is read back with sched_total. scratch holds
// scratch_ints ints of the caller's (at least P + 1) for per-warp counters.
// Every thread of the block must call it; it synchronises the block.
//
// Placement is a stable counting sort: W warps each own a contiguous range of
// sequence indices; per value v, warp w's sequences go after those of value
// v in the ranges of warps 0..w-1, and inside a warp's range in index order
// (ranks among 32 lanes from __match_any_sync). No position depends on the
// order in which threads happen to run.
template <class CountFn>
__device__ void build_sched(const Sched& s, int n, int P, int H, bool causal, bool top_first,
                            CountFn count, int* scratch, int scratch_ints) {
  const int V = P + 1;  // values 0..P
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = max(1, min(static_cast<int>(blockDim.x >> 5), scratch_ints / V));
  const int span = (n + W - 1) / W;  // sequences per placing warp
  for (int i = threadIdx.x; i < W * V; i += blockDim.x) scratch[i] = 0;
  __syncthreads();
  // c_b, parked in pre[b] until the placement is done, and per-warp counts
  for (int b = threadIdx.x; b < n; b += blockDim.x) {
    const int c = min(count(b), P);
    s.pre[b] = c;
    atomicAdd(&scratch[(b / span) * V + c], 1);
  }
  __syncthreads();
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    int t = 0;
    for (int w = 0; w < W; ++w) t += scratch[w * V + v];
    s.hist[v] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // where value v starts in sorted (largest first) = sequences with more than v levels
    int above = 0;
    for (int v = P; v >= 0; --v) {
      const int h = s.hist[v];
      s.hist[v] = above;
      s.kcount[v] = above;
      above += h;
    }
    // causal: the t-th level visited is P - 1 - t (top_first) or t
    int total = 0;
    for (int t = 0; t < P; ++t) {
      s.start[t] = total;
      total += H * s.kcount[top_first ? P - 1 - t : t];
    }
    s.start[P] = total;
  }
  __syncthreads();
  // per value, the first position of each warp's sequences
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    int run = s.hist[v];
    for (int w = 0; w < W; ++w) {
      const int t = scratch[w * V + v];
      scratch[w * V + v] = run;
      run += t;
    }
  }
  __syncthreads();
  if (warp < W) {
    int* next = scratch + warp * V;
    const int hi = min(n, (warp + 1) * span);
    for (int c0 = warp * span; c0 < hi; c0 += 32) {
      const int b = c0 + lane;
      const int v = b < hi ? s.pre[b] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, v);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (v >= 0) s.sorted[next[v] + rank] = b;
      __syncwarp();
      if (v >= 0 && rank == 0) next[v] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  if (!causal) {
    // rank r has the c levels with kcount[c] <= r < kcount[c - 1]
    for (int r = threadIdx.x; r < n; r += blockDim.x) {
      int lo = 0, hi = P;  // the number of v in [0, P) with kcount[v] > r (non-increasing)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s.kcount[mid] > r) lo = mid + 1;
        else hi = mid;
      }
      s.pre[r + 1] = H * lo;
    }
    __syncthreads();
    if (threadIdx.x < 32) scan_counts_warp(s.pre, n, threadIdx.x);
    __syncthreads();
  }
}

__device__ __forceinline__ int sched_total(const Sched& s, int n, int P, bool causal) {
  return causal ? s.start[P] : s.pre[n];
}

// The largest index i in [0, m) with a[i] <= x (a non-decreasing).
__device__ __forceinline__ int last_le(const int* a, int m, int x) {
  int lo = 0, hi = m - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Item -> (sequence b, head h, level) of the schedule. In the forward the
// causal levels are visited from the top (level = P - 1 - t), in the
// backward from 0 (top_first = false).
__device__ __forceinline__ void sched_decode(const Sched& s, int n, int P, int H, bool causal,
                                             bool top_first, int item, int& b, int& h,
                                             int& level) {
  if (causal) {
    const int t = last_le(s.start, P, item);
    const int r = item - s.start[t];
    const int lv = top_first ? P - 1 - t : t;
    const int rank = r / H;
    h = r - rank * H;
    b = s.sorted[rank];
    level = lv;
  } else {
    const int r = last_le(s.pre, n, item);
    const int rem = item - s.pre[r];
    const int np = (s.pre[r + 1] - s.pre[r]) / H;
    h = rem / np;
    level = rem - h * np;
    b = s.sorted[r];
  }
}

// Padded D / lse2 rows per (batch, head) plane: every sequence's rows fit
// from its s.pst on, whatever the (clamped) offsets hold. rows_q: query rows
// per plane; B: sequences.
inline int var_padded_rows(bool packed, int B, int rows_q) {
  if (packed) return ((rows_q + kTile - 1) / kTile + B + 1) * kTile;
  return (rows_q + kTile - 1) / kTile * kTile;
}

}  // namespace fa

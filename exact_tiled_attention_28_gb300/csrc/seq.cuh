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
// stays inside the tensors (a separate check reports them).
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
    s.nk = g.Nk;
    s.pst = 0;
  }
  return s;
}

// Padded D / lse2 rows per (batch, head) plane: every sequence's rows fit
// from its s.pst on, whatever the (clamped) offsets hold. rows_q: query rows
// per plane; B: sequences.
inline int var_padded_rows(bool packed, int B, int rows_q) {
  if (packed) return ((rows_q + kTile - 1) / kTile + B + 1) * kTile;
  return (rows_q + kTile - 1) / kTile * kTile;
}

}  // namespace fa

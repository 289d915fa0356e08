"""fp64 CPU oracle for exact scaled-dot-product attention and its gradients.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module. The CUDA path never calls it, and it calls nothing of the CUDA path.

What it computes
----------------
The pages agree that the tiled method reaches *exactly* the result of
standard attention, only with less memory traffic ("flashattention-2"
glossary, definition and the "Performance Comparison" table column "Exact?";
"FlashAttention-2 paper", section "What changed and what did not"). So the
oracle is that standard definition written out with materialised score and
probability matrices ("Flash Attention v2" notes, section "Flash Attention v1:
Recap", the standard attention steps; the 1/sqrt(d) scaling and the
max-subtracted exponent from "Detailed Algorithm Comparison", forward pass):

    S = scale * Q K^T            (Q: Nq rows, K and V: Nk rows; when causal,
                                  query i sees key j only if j <= i + Nk - Nq)
    m_i = max_j S_ij
    P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)
    O = P V
    LSE_i = m_i + ln sum_j exp(S_ij - m_i)      (natural log)

The backward is the standard calculus of that definition (the notes'
"Backward Pass Computation" section prints a diagonal-only softmax Jacobian,
which is wrong; the full Jacobian is used):

    dV = P^T dO
    dP = dO V^T
    D_i = sum_j P_ij dP_ij
    dS = P o (dP - D 1^T)
    dQ = scale * dS K
    dK = scale * dS^T Q

Everything is float64. Inputs are the exact float64 values of the bf16 inputs.

Unequal lengths and packed batches
----------------------------------
The pages state the method for one sequence length N. They also speak of
serving with batches of requests of different lengths ("Flash Attention v2"
notes, "Performance Comparison: v1 vs v2", continuous batching, and
"Detailed Differences" 4, "Batch and Sequence Length Support"), but fix no
convention for them. The readings taken here:

* Nq query rows may attend to Nk != Nq keys. The causal mask is aligned at
  the bottom right: query i sees key j when j <= i + (Nk - Nq), so the last
  query sees every key (new tokens come after the cached ones). With
  Nq = Nk this is the usual top-left rule.
* A query row with no visible key (causal with Nq > Nk, or Nk = 0) has
  O = 0 and LSE = -inf, and contributes nothing to any gradient.
* A packed batch holds B sequences back to back along the token axis:
  q is [Tq, H, d], k and v are [Tk, H, d], and sequence b owns query rows
  cu_q[b] .. cu_q[b+1]-1 and key rows cu_k[b] .. cu_k[b+1]-1. Each
  (sequence, head) is an independent attention of the kind above; LSE is
  [H, Tq].

Rows of the definition are independent, so a head is evaluated in stripes of
at most ``ROW_STRIPE`` query rows to bound memory (one stripe of S at
N = 32768 is 256 MiB). dK and dV are sums over query rows; the stripes add
their partial sums in row order. ``rows=`` evaluates only the listed query
rows, which is how the full-size checks sample outputs one by one.

Parity is pinned by the ``tests/test_oracle_*.py`` suite: multi-precision
brute force, PyTorch's float64 attention and autograd, central finite
differences, closed forms and invariants.
"""

from __future__ import annotations

import numpy as np

ROW_STRIPE = 1024


def _scores(q_rows, k, rows, causal, scale, n_q):
    """S for the given query rows: scale * q_rows k^T, causally masked with
    the bottom-right alignment (query i of n_q sees key j <= i + Nk - n_q)."""
    S = scale * (q_rows @ k.T)
    if causal:
        keys = np.arange(k.shape[0])
        S = np.where(keys[None, :] > rows[:, None] + (k.shape[0] - n_q), -np.inf, S)
    return S


def _softmax_rows(S):
    """Row softmax of S and its log-sum-exp, max-subtracted. A row with no
    finite entry (no visible key) gets P = 0 and LSE = -inf."""
    if S.shape[1] == 0:
        return np.zeros(S.shape), np.full(S.shape[0], -np.inf)
    m = S.max(axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.exp(S - m_safe[:, None])
    l = E.sum(axis=1)
    P = E / np.where(empty, 1.0, l)[:, None]
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, l)))
    return P, lse


def _stripes(rows):
    for s in range(0, rows.shape[0], ROW_STRIPE):
        yield rows[s:s + ROW_STRIPE]


def _check_head(q, k, v, scale):
    if q.ndim != 2 or k.ndim != 2 or v.shape != k.shape or k.shape[1] != q.shape[1]:
        raise ValueError("expected q [Nq, d] and k, v of one shape [Nk, d]")
    if not np.isfinite(scale):
        raise ValueError("scale must be finite")


def head_forward(q, k, v, causal, scale, rows=None):
    """Forward of one head.

    q: float64 [Nq, d]; k, v: float64 [Nk, d]. Returns (O [R, d], LSE [R])
    for the R query rows in ``rows`` (all rows by default), in that order.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    _check_head(q, k, v, scale)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.empty((rows.shape[0], q.shape[1]))
    lse = np.empty(rows.shape[0])
    pos = 0
    for r in _stripes(rows):
        P, lse_r = _softmax_rows(_scores(q[r], k, r, causal, scale, q.shape[0]))
        O[pos:pos + r.shape[0]] = P @ v
        lse[pos:pos + r.shape[0]] = lse_r
        pos += r.shape[0]
    return O, lse


def head_backward(q, k, v, do, causal, scale, rows=None):
    """Backward of one head for the loss sum(O o dO).

    Returns (dQ [R, d] for the listed query rows, dK [Nk, d], dV [Nk, d]) where
    dK and dV are the contributions of the listed query rows (the full
    gradients when ``rows`` is every row, the default).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    _check_head(q, k, v, scale)
    if do.shape != q.shape:
        raise ValueError("dO must have the shape of q")
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    dQ = np.empty((rows.shape[0], q.shape[1]))
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    pos = 0
    for r in _stripes(rows):
        P, _ = _softmax_rows(_scores(q[r], k, r, causal, scale, q.shape[0]))
        dV += P.T @ do[r]
        dP = do[r] @ v.T
        D = (P * dP).sum(axis=1)
        dS = P * (dP - D[:, None])
        dQ[pos:pos + r.shape[0]] = scale * (dS @ k)
        dK += scale * (dS.T @ q[r])
        pos += r.shape[0]
    return dQ, dK, dV


def head_probabilities(q, k, causal, scale):
    """The full probability matrix P [Nq, Nk] of one head (small sizes only)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    rows = np.arange(q.shape[0])
    P, _ = _softmax_rows(_scores(q, k, rows, causal, scale, q.shape[0]))
    return P


def attention_forward(q, k, v, causal, scale):
    """Forward over float64 q [B, H, Nq, d] and k, v [B, H, Nk, d]:
    (O [B,H,Nq,d], LSE [B,H,Nq])."""
    B, H, N, d = q.shape
    O = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            O[b, h], lse[b, h] = head_forward(q[b, h], k[b, h], v[b, h], causal, scale)
    return O, lse


def attention_backward(q, k, v, do, causal, scale):
    """Backward over float64 q, do [B, H, Nq, d] and k, v [B, H, Nk, d]:
    (dQ, dK, dV)."""
    dQ = np.empty(q.shape)
    dK = np.empty(k.shape)
    dV = np.empty(v.shape)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h] = head_backward(
                q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
    return dQ, dK, dV



def _check_packed(q, k, v, cu_q, cu_k):
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_k = np.asarray(cu_k, dtype=np.int64)
    if q.ndim != 3 or k.ndim != 3 or v.shape != k.shape or k.shape[1:] != q.shape[1:]:
        raise ValueError("expected q [Tq, H, d] and k, v of one shape [Tk, H, d]")
    if (cu_q.ndim != 1 or cu_q.shape != cu_k.shape or cu_q.shape[0] < 2
            or cu_q[0] != 0 or cu_k[0] != 0 or np.any(np.diff(cu_q) < 0)
            or np.any(np.diff(cu_k) < 0) or cu_q[-1] != q.shape[0] or cu_k[-1] != k.shape[0]):
        raise ValueError("cu_q, cu_k must be non-decreasing prefix offsets from 0 to Tq, Tk")
    return cu_q, cu_k


def varlen_forward(q, k, v, cu_q, cu_k, causal, scale):
    """Forward of a packed batch: q [Tq, H, d], k, v [Tk, H, d] float64,
    sequence b on rows cu_q[b]..cu_q[b+1]-1 and cu_k[b]..cu_k[b+1]-1.
    Returns (O [Tq, H, d], LSE [H, Tq])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    cu_q, cu_k = _check_packed(q, k, v, cu_q, cu_k)
    Tq, H, d = q.shape
    O = np.zeros((Tq, H, d))
    lse = np.empty((H, Tq))
    for b in range(cu_q.shape[0] - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if q1 == q0:
            continue
        for h in range(H):
            O[q0:q1, h], lse[h, q0:q1] = head_forward(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h],
                                                      causal, scale)
    return O, lse


def varlen_backward(q, k, v, do, cu_q, cu_k, causal, scale):
    """Backward of a packed batch (see varlen_forward): (dQ [Tq,H,d],
    dK [Tk,H,d], dV [Tk,H,d])."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    cu_q, cu_k = _check_packed(q, k, v, cu_q, cu_k)
    if do.shape != q.shape:
        raise ValueError("dO must have the shape of q")
    dQ = np.zeros(q.shape)
    dK = np.zeros(k.shape)
    dV = np.zeros(v.shape)
    for b in range(cu_q.shape[0] - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if q1 == q0:
            continue
        for h in range(q.shape[1]):
            dQ[q0:q1, h], dK[k0:k1, h], dV[k0:k1, h] = head_backward(
                q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], do[q0:q1, h], causal, scale)
    return dQ, dK, dV

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

    S = scale * Q K^T            (entries with key index > query index are -inf
                                  when causal: top-left aligned, Nq = Nk)
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


def _scores(q_rows, k, rows, causal, scale):
    """S for the given query rows: scale * q_rows k^T, causally masked."""
    S = scale * (q_rows @ k.T)
    if causal:
        keys = np.arange(k.shape[0])
        S = np.where(keys[None, :] > rows[:, None], -np.inf, S)
    return S


def _softmax_rows(S):
    """Row softmax of S and its log-sum-exp, max-subtracted."""
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])
    l = E.sum(axis=1)
    return E / l[:, None], m + np.log(l)


def _stripes(rows):
    for s in range(0, rows.shape[0], ROW_STRIPE):
        yield rows[s:s + ROW_STRIPE]


def _check_head(q, k, v, scale):
    if q.ndim != 2 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("expected q, k, v of one shape [N, d]")
    if q.shape[0] < 1:
        raise ValueError("N must be at least 1")
    if not np.isfinite(scale):
        raise ValueError("scale must be finite")


def head_forward(q, k, v, causal, scale, rows=None):
    """Forward of one head.

    q, k, v: float64 [N, d]. Returns (O [R, d], LSE [R]) for the R query rows
    in ``rows`` (all rows by default), in that order.
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
        P, lse_r = _softmax_rows(_scores(q[r], k, r, causal, scale))
        O[pos:pos + r.shape[0]] = P @ v
        lse[pos:pos + r.shape[0]] = lse_r
        pos += r.shape[0]
    return O, lse


def head_backward(q, k, v, do, causal, scale, rows=None):
    """Backward of one head for the loss sum(O o dO).

    Returns (dQ [R, d] for the listed query rows, dK [N, d], dV [N, d]) where
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
        P, _ = _softmax_rows(_scores(q[r], k, r, causal, scale))
        dV += P.T @ do[r]
        dP = do[r] @ v.T
        D = (P * dP).sum(axis=1)
        dS = P * (dP - D[:, None])
        dQ[pos:pos + r.shape[0]] = scale * (dS @ k)
        dK += scale * (dS.T @ q[r])
        pos += r.shape[0]
    return dQ, dK, dV


def head_probabilities(q, k, causal, scale):
    """The full probability matrix P [N, N] of one head (small N only)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    rows = np.arange(q.shape[0])
    P, _ = _softmax_rows(_scores(q, k, rows, causal, scale))
    return P


def attention_forward(q, k, v, causal, scale):
    """Forward over [B, H, N, d] float64 arrays: (O [B,H,N,d], LSE [B,H,N])."""
    B, H, N, d = q.shape
    O = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            O[b, h], lse[b, h] = head_forward(q[b, h], k[b, h], v[b, h], causal, scale)
    return O, lse


def attention_backward(q, k, v, do, causal, scale):
    """Backward over [B, H, N, d] float64 arrays: (dQ, dK, dV)."""
    dQ = np.empty(q.shape)
    dK = np.empty(q.shape)
    dV = np.empty(q.shape)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h] = head_backward(
                q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
    return dQ, dK, dV


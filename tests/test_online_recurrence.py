"""The tiled online-softmax recurrence that the CUDA forward implements,
restated on the CPU in fp64 and compared with the oracle.

The recurrence is the one in the "Flash Attention v2" notes, "Detailed
Algorithm Comparison", forward pass: per query block keep a running row max m
and running sum l; for each key/value block, m_new = max(m, rowmax(S)),
P = exp(S - m_new), l = exp(m - m_new) l + rowsum(P),
O = exp(m - m_new) O + P V. The page writes O without the final division;
the exact softmax needs O / l at the end (read that way). The "flashattention-2"
glossary's improvements table ("Causal Masking": fully masked tiles skipped)
gives the causal tile skip, and the "FlashAttention-2 paper" digest ("delays
and batches the rescaling") the deferred rescale, here as a threshold tau: the
running maximum used for the exponent is only raised when the true maximum
exceeds it by more than tau, which is exact in real arithmetic because O and l
are always scaled by the same factor.

This is a test of the recurrence, not the oracle: it pins the arithmetic the
GPU kernel performs to the plain definition, in exact-enough fp64.
"""

import math

import numpy as np
import pytest

import oracle

from . import pins


def tiled_forward(q, k, v, causal, scale, Br, Bc, tau=0.0, reverse_kv=False):
    N, d = q.shape
    O = np.zeros((N, d))
    lse = np.zeros(N)
    for i0 in range(0, N, Br):
        rows = np.arange(i0, min(i0 + Br, N))
        m = np.full(rows.shape[0], -np.inf)
        l = np.zeros(rows.shape[0])
        acc = np.zeros((rows.shape[0], d))
        last = N if not causal else min(N, rows[-1] + 1)  # skip fully masked key blocks
        blocks = list(range(0, last, Bc))
        if reverse_kv:
            blocks = blocks[::-1]
        for j0 in blocks:
            cols = np.arange(j0, min(j0 + Bc, N))
            S = scale * (q[rows] @ k[cols].T)
            if causal:
                S = np.where(cols[None, :] > rows[:, None], -np.inf, S)
            mt = S.max(axis=1)
            grow = mt > m + tau           # raise the reference max only past tau
            m_new = np.where(grow, mt, m)
            alpha = np.where(np.isneginf(m), 0.0, np.exp(np.where(np.isneginf(m), 0.0, m - m_new)))
            P = np.exp(S - m_new[:, None])
            l = alpha * l + P.sum(axis=1)
            acc = alpha[:, None] * acc + P @ v[cols]
            m = m_new
        O[rows] = acc / l[:, None]
        lse[rows] = m + np.log(l)
    return O, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,Br,Bc", [(1, 4, 4), (37, 8, 8), (37, 8, 5), (64, 16, 16), (50, 7, 16)])
@pytest.mark.parametrize("tau", [0.0, 8.0 * math.log(2.0)])
def test_tiled_equals_definition(causal, N, Br, Bc, tau):
    t = pins.rand_head(71 + N, N, 16)
    scale = 1.0 / math.sqrt(16)
    O, lse = oracle.head_forward(t["q"], t["k"], t["v"], causal, scale)
    Ot, lset = tiled_forward(t["q"], t["k"], t["v"], causal, scale, Br, Bc, tau)
    assert np.max(np.abs(Ot - O)) < 1e-12
    assert np.max(np.abs(lset - lse)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_key_block_order_is_free(causal):
    """The notes' "reversed" key/value iteration gives the same result: the
    order of key blocks is a free scheduling choice."""
    t = pins.rand_head(90, 61, 8)
    a = tiled_forward(t["q"], t["k"], t["v"], causal, 0.4, 16, 16)
    b = tiled_forward(t["q"], t["k"], t["v"], causal, 0.4, 16, 16, reverse_kv=True)
    assert np.max(np.abs(a[0] - b[0])) < 1e-12
    assert np.max(np.abs(a[1] - b[1])) < 1e-12


def test_key_splits_merged_by_log_sum_exp():
    """Splitting the keys into contiguous ranges, attending to each range
    alone and merging the parts with weights exp(LSE_s - LSE), LSE = ln sum_s
    exp(LSE_s), gives the whole attention: the identity the decode path's
    split-KV merge rests on. Ranges that no query can see (LSE_s = -inf)
    weigh nothing."""
    t = pins._head_pair(131, 3, 700, 16)
    for causal in (False, True):
        O, lse = oracle.head_forward(t["q"], t["k"], t["v"], causal, 0.3)
        parts = []
        for k0, k1 in ((0, 128), (128, 300), (300, 301), (301, 700)):
            kk, vv = t["k"][:k1], t["v"][:k1]
            # the range's own attention: keys outside [k0, k1) masked out, with
            # the causal alignment of the whole key set
            Os, ls = oracle.head_forward(t["q"], kk[k0:], vv[k0:], False, 0.3)
            if causal:
                keep = np.arange(k0, k1)[None, :] <= np.arange(3)[:, None] + 700 - 3
                S = 0.3 * t["q"] @ kk[k0:].T
                S = np.where(keep, S, -np.inf)
                m = np.max(S, axis=1, keepdims=True)
                fin = np.isfinite(m[:, 0])
                E = np.exp(S - np.where(np.isfinite(m), m, 0.0))
                l = E.sum(axis=1)
                Os = np.where(fin[:, None], (E @ vv[k0:]) / np.where(l > 0, l, 1.0)[:, None], 0.0)
                with np.errstate(divide="ignore"):
                    ls = np.where(fin, m[:, 0] + np.log(np.where(l > 0, l, 1.0)), -np.inf)
            parts.append((Os, ls))
        L = np.stack([p[1] for p in parts])
        M = L.max(axis=0)
        W = np.exp(L - M)
        lse_m = M + np.log(W.sum(axis=0))
        O_m = sum(w[:, None] * p[0] for w, p in zip(W, parts)) / W.sum(axis=0)[:, None]
        assert np.max(np.abs(O_m - O)) < 1e-12 and np.max(np.abs(lse_m - lse)) < 1e-12

"""Host-side check of the index arithmetic the kernels use to place the
sequences of a packed batch (csrc/seq.cuh: the clamped offsets and the
backward's padded D / lse2 rows): whatever the offsets hold, every row a
kernel touches lies inside its buffer, and well-formed offsets give
non-overlapping padded rows. The arithmetic is restated here in Python; the
GPU tests then run the kernels on well-formed and malformed offsets."""

import numpy as np

TILE = 128


def seq_of(b, cu_q, cu_k, rows_q, rows_k, max_q, max_k):
    q0 = min(max(int(cu_q[b]), 0), rows_q)
    q1 = min(max(int(cu_q[b + 1]), q0), rows_q)
    k0 = min(max(int(cu_k[b]), 0), rows_k)
    k1 = min(max(int(cu_k[b + 1]), k0), rows_k)
    pst = ((q0 + TILE - 1) // TILE + b) * TILE
    return q0, k0, min(q1 - q0, max_q), min(k1 - k0, max_k), pst


def padded_rows(B, rows_q):
    return ((rows_q + TILE - 1) // TILE + B + 1) * TILE


def test_every_access_stays_in_bounds():
    rng = np.random.default_rng(0)
    for trial in range(20000):
        B = int(rng.integers(1, 9))
        rows_q, rows_k = int(rng.integers(1, 3000)), int(rng.integers(1, 3000))
        max_q, max_k = int(rng.integers(1, 3000)), int(rng.integers(1, 3000))
        if trial % 2:  # arbitrary, possibly malformed offsets
            cu_q = rng.integers(-100, rows_q + 300, size=B + 1)
            cu_k = rng.integers(-100, rows_k + 300, size=B + 1)
        else:
            cu_q = np.concatenate([[0], np.sort(rng.integers(0, rows_q + 1, B - 1)), [rows_q]])
            cu_k = np.concatenate([[0], np.sort(rng.integers(0, rows_k + 1, B - 1)), [rows_k]])
        lpad = padded_rows(B, rows_q)
        spans = []
        for b in range(B):
            q0, k0, nq, nk, pst = seq_of(b, cu_q, cu_k, rows_q, rows_k, max_q, max_k)
            assert 0 <= nq and q0 + nq <= rows_q and 0 <= nk and k0 + nk <= rows_k
            assert pst % TILE == 0  # 512-byte aligned tiles of fp32 rows
            if nq:
                end = pst + -(-nq // TILE) * TILE
                assert end <= lpad
                spans.append((pst, end))
        if trial % 2 == 0:  # well-formed: the sequences' padded rows do not overlap
            spans.sort()
            assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))

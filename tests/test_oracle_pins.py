"""The fp64 oracle against pins that do not come from the oracle itself.

Runs on the CPU only (``-m "not gpu"``).
"""

import math

import numpy as np
import pytest

import oracle
from oracle import attention as orc

from . import pins

pytest.importorskip("mpmath")
pytest.importorskip("torch")


def oracle_fwd(q, k, v, causal, scale):
    return oracle.head_forward(q, k, v, causal, scale)


def oracle_bwd(q, k, v, do, causal, scale):
    return oracle.head_backward(q, k, v, do, causal, scale)


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    ok, msg = check(oracle_fwd, oracle_bwd)
    assert ok, msg


@pytest.mark.parametrize("check", pins.VARLEN_CHECKS, ids=lambda c: c.__name__)
def test_oracle_varlen_pin(check):
    ok, msg = check(oracle.varlen_forward, oracle.varlen_backward)
    assert ok, msg


def test_rows_of_p_sum_to_one():
    for causal in (False, True):
        t = pins.rand_head(51, 45, 8)
        P = oracle.head_probabilities(t["q"], t["k"], causal, 0.5)
        assert np.all(P >= 0)
        assert np.max(np.abs(P.sum(axis=1) - 1.0)) < 1e-12
        if causal:
            assert np.all(np.triu(P, 1) == 0.0)


def test_d_identity():
    """sum_j P_ij dP_ij equals sum_c dO_ic O_ic because O = P V; the GPU
    backward pre-pass relies on the second form."""
    for causal in (False, True):
        t = pins.rand_head(52, 40, 8)
        P = oracle.head_probabilities(t["q"], t["k"], causal, 0.4)
        O, _ = oracle.head_forward(t["q"], t["k"], t["v"], causal, 0.4)
        dP = t["do"] @ t["v"].T
        assert np.max(np.abs((P * dP).sum(axis=1) - (t["do"] * O).sum(axis=1))) < 1e-12


def test_row_subsets_and_stripes(monkeypatch):
    """Evaluating a subset of rows, or the rows in small stripes, reproduces
    the rows of the full evaluation; dK and dV from all stripes add up to the
    full gradient."""
    t = pins.rand_head(53, 50, 8)
    for causal in (False, True):
        O, lse = oracle.head_forward(t["q"], t["k"], t["v"], causal, 0.3)
        dQ, dK, dV = oracle.head_backward(t["q"], t["k"], t["v"], t["do"], causal, 0.3)
        rows = np.array([0, 7, 49, 13])
        Os, lses = oracle.head_forward(t["q"], t["k"], t["v"], causal, 0.3, rows=rows)
        dQs, _, _ = oracle.head_backward(t["q"], t["k"], t["v"], t["do"], causal, 0.3, rows=rows)
        assert np.max(np.abs(Os - O[rows])) < 1e-14
        assert np.max(np.abs(lses - lse[rows])) < 1e-14
        assert np.max(np.abs(dQs - dQ[rows])) < 1e-14
        monkeypatch.setattr(orc, "ROW_STRIPE", 7)
        O7, lse7 = oracle.head_forward(t["q"], t["k"], t["v"], causal, 0.3)
        dQ7, dK7, dV7 = oracle.head_backward(t["q"], t["k"], t["v"], t["do"], causal, 0.3)
        monkeypatch.undo()
        for a, b in ((O7, O), (lse7, lse), (dQ7, dQ), (dK7, dK), (dV7, dV)):
            assert np.max(np.abs(a - b)) < 1e-12


def test_batched_wrappers_match_heads():
    B, H, N, d = 2, 3, 20, 4
    x = {n: np.stack([np.stack([pins.rand_head(60 + b, N, d, (n,), b=b, h=h)[n]
                                for h in range(H)]) for b in range(B)])
         for n in ("q", "k", "v", "do")}
    O, lse = oracle.attention_forward(x["q"], x["k"], x["v"], True, 0.5)
    dQ, dK, dV = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], True, 0.5)
    for b in range(B):
        for h in range(H):
            o1, l1 = oracle.head_forward(x["q"][b, h], x["k"][b, h], x["v"][b, h], True, 0.5)
            g = oracle.head_backward(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["do"][b, h],
                                     True, 0.5)
            assert np.array_equal(O[b, h], o1) and np.array_equal(lse[b, h], l1)
            assert np.array_equal(dQ[b, h], g[0]) and np.array_equal(dK[b, h], g[1])
            assert np.array_equal(dV[b, h], g[2])


def test_oracle_rejects_bad_arguments():
    t = pins.rand_head(61, 4, 2)
    with pytest.raises(ValueError):
        oracle.head_forward(t["q"], t["k"][:3], t["v"], False, 1.0)
    with pytest.raises(ValueError):
        oracle.head_forward(t["q"], t["k"][:, :1], t["v"][:, :1], False, 1.0)
    x, cu_q, cu_k = pins.packed_inputs(62, [2, 3], [3, 1], 1, 2)
    for bad_q, bad_k in (([0, 2, 4], cu_k), ([1, 2, 5], cu_k), ([0, 3, 2], cu_k),
                         (cu_q, [0, 3])):
        with pytest.raises(ValueError):
            oracle.varlen_forward(x["q"], x["k"], x["v"], bad_q, bad_k, False, 1.0)
    with pytest.raises(ValueError):
        oracle.head_forward(t["q"], t["k"], t["v"], False, math.inf)
    with pytest.raises(ValueError):
        oracle.head_backward(t["q"], t["k"], t["v"], t["do"][:, :1], False, 1.0)

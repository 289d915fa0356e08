"""Pin checks for an exact-attention implementation on the CPU.

Each ``check_*`` takes a per-head forward ``fwd(q, k, v, causal, scale)
-> (O, LSE)`` and backward ``bwd(q, k, v, do, causal, scale) -> (dQ, dK, dV)``
(float64 [N, d] arrays) and returns ``(ok, message)``. The oracle tests run
them on the oracle; the planted-mistake test runs them on deliberately broken
copies of it and requires each copy to fail at least one check.

None of them restates the oracle's formulas: they compare against
multi-precision brute force, PyTorch's float64 attention and autograd,
finite differences, closed forms and invariants that the definition of exact
attention fixes.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

from exact_tiled_attention_28_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_head(seed, N, d, tensors=("q", "k", "v", "do"), b=0, h=0):
    return inputs.head_inputs_f64(seed, b, h, N, d, tensors)


def _close(a, b, atol, rtol=0.0):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.shape != b.shape:
        return False, f"shape {a.shape} vs {b.shape}"
    if not np.all(np.isfinite(a)):
        return False, "non-finite values"
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    if np.all(err <= lim):
        return True, ""
    i = np.unravel_index(np.argmax(err - lim), err.shape)
    return False, f"max excess at {i}: {a[i]} vs {b[i]}"


def _all(results):
    for ok, msg in results:
        if not ok:
            return False, msg
    return True, ""


# --------------------------------------------------------------------------
# hand-worked closed-form example (tests/golden/hand_worked_n2_d1.json)

def check_golden(fwd, bwd):
    with open(os.path.join(GOLDEN, "hand_worked_n2_d1.json")) as f:
        g = json.load(f)
    q, k, v, do = (np.array(g[t], np.float64) for t in ("q", "k", "v", "do"))
    res = []
    for causal, key in ((False, "noncausal"), (True, "causal")):
        want = {n: np.array([[eval(e, {"math": math})] for e in g[key][n]]) for n in ("O", "dV")}
        want_lse = np.array([eval(e, {"math": math}) for e in g[key]["LSE"]])
        O, lse = fwd(q, k, v, causal, g["scale"])
        _, _, dV = bwd(q, k, v, do, causal, g["scale"])
        res += [_close(O, want["O"], 1e-14), _close(lse, want_lse, 1e-14),
                _close(dV, want["dV"], 1e-14)]
    return _all(res)


# --------------------------------------------------------------------------
# multi-precision brute force (mpmath, 40 digits): forward from the definition,
# backward by central differences of the multi-precision loss

def _mp_forward(q, k, v, causal, scale):
    import mpmath as mp
    N, d = len(q), len(q[0])
    O, L = [], []
    for i in range(N):
        keys = [j for j in range(N) if not (causal and j > i)]
        s = {j: scale * mp.fsum(q[i][c] * k[j][c] for c in range(d)) for j in keys}
        z = mp.fsum(mp.exp(s[j]) for j in keys)
        O.append([mp.fsum(mp.exp(s[j]) * v[j][c] for j in keys) / z for c in range(d)])
        L.append(mp.log(z))
    return O, L


def check_multiprecision(fwd, bwd):
    import mpmath as mp
    res = []
    with mp.workdps(40):
        for seed, N, d, causal in ((1, 1, 2, False), (2, 3, 2, False), (3, 3, 2, True),
                                   (4, 5, 3, True), (5, 4, 1, False)):
            t = rand_head(seed, N, d)
            scale = 1.0 / math.sqrt(d) * 1.7
            mq, mk, mv, mdo = ([[mp.mpf(float(x)) for x in row] for row in t[n]]
                               for n in ("q", "k", "v", "do"))
            Omp, Lmp = _mp_forward(mq, mk, mv, causal, mp.mpf(scale))
            O, lse = fwd(t["q"], t["k"], t["v"], causal, scale)
            res.append(_close(O, np.array([[float(x) for x in r] for r in Omp]), 1e-13))
            res.append(_close(lse, np.array([float(x) for x in Lmp]), 1e-13))

            def loss(mats):
                Om, _ = _mp_forward(mats[0], mats[1], mats[2], causal, mp.mpf(scale))
                return mp.fsum(Om[i][c] * mdo[i][c] for i in range(N) for c in range(d))

            h = mp.mpf("1e-15")
            grads = []
            for which in range(3):
                g = np.zeros((N, d))
                for i in range(N):
                    for c in range(d):
                        mats = [[row[:] for row in m] for m in (mq, mk, mv)]
                        x0 = mats[which][i][c]
                        mats[which][i][c] = x0 + h
                        lp = loss(mats)
                        mats[which][i][c] = x0 - h
                        lm = loss(mats)
                        g[i, c] = float((lp - lm) / (2 * h))
                grads.append(g)
            dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], causal, scale)
            for got, want in zip((dQ, dK, dV), grads):
                res.append(_close(got, want, 1e-12))
    return _all(res)


# --------------------------------------------------------------------------
# PyTorch float64 scaled_dot_product_attention and autograd (library routine)

def check_torch_float64(fwd, bwd):
    import torch
    import torch.nn.functional as F
    res = []
    for seed, N, d, causal in ((11, 37, 16, False), (12, 37, 16, True), (13, 70, 8, True)):
        t = rand_head(seed, N, d)
        scale = 1.0 / math.sqrt(d)
        tq, tk, tv = (torch.tensor(t[n], dtype=torch.float64, requires_grad=True)
                      for n in ("q", "k", "v"))
        out = F.scaled_dot_product_attention(tq[None], tk[None], tv[None],
                                             is_causal=causal, scale=scale)[0]
        out.backward(torch.tensor(t["do"], dtype=torch.float64))
        s = scale * (tq.detach() @ tk.detach().T)
        if causal:
            s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        lse_t = torch.logsumexp(s, dim=1)
        O, lse = fwd(t["q"], t["k"], t["v"], causal, scale)
        dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], causal, scale)
        res += [_close(O, out.detach().numpy(), 1e-12), _close(lse, lse_t.numpy(), 1e-12),
                _close(dQ, tq.grad.numpy(), 1e-11), _close(dK, tk.grad.numpy(), 1e-11),
                _close(dV, tv.grad.numpy(), 1e-11)]
    return _all(res)


# --------------------------------------------------------------------------
# float64 central differences of the forward under test

def check_finite_differences(fwd, bwd):
    res = []
    for seed, N, d, causal in ((21, 9, 4, False), (22, 9, 4, True)):
        t = rand_head(seed, N, d)
        scale = 0.5
        dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], causal, scale)
        h = 1e-6
        for name, got in (("q", dQ), ("k", dK), ("v", dV)):
            g = np.zeros((N, d))
            for i in range(N):
                for c in range(d):
                    x = {n: t[n].copy() for n in ("q", "k", "v")}
                    x[name][i, c] += h
                    lp = np.sum(fwd(x["q"], x["k"], x["v"], causal, scale)[0] * t["do"])
                    x[name][i, c] -= 2 * h
                    lm = np.sum(fwd(x["q"], x["k"], x["v"], causal, scale)[0] * t["do"])
                    g[i, c] = (lp - lm) / (2 * h)
            res.append(_close(got, g, 1e-7, 1e-6))
    return _all(res)


# --------------------------------------------------------------------------
# closed forms

def check_single_token(fwd, bwd):
    """N = 1: O = V, LSE = scale q.k, dQ = dK = 0, dV = dO."""
    res = []
    for causal in (False, True):
        t = rand_head(31, 1, 8)
        scale = 0.3
        O, lse = fwd(t["q"], t["k"], t["v"], causal, scale)
        dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], causal, scale)
        res += [_close(O, t["v"], 1e-15), _close(lse, scale * t["q"] @ t["k"][0], 1e-15),
                _close(dQ, np.zeros((1, 8)), 1e-15), _close(dK, np.zeros((1, 8)), 1e-15),
                _close(dV, t["do"], 1e-15)]
    return _all(res)


def check_constant_v(fwd, bwd):
    """Every V row equal to c gives every O row equal to c."""
    res = []
    for causal in (False, True):
        t = rand_head(32, 23, 6)
        c = t["v"][5]
        v = np.tile(c, (23, 1))
        O, _ = fwd(t["q"], t["k"], v, causal, 0.4)
        res.append(_close(O, np.tile(c, (23, 1)), 1e-13))
    return _all(res)


def check_zero_scale(fwd, bwd):
    """scale = 0: O_i is the mean of the visible V rows, LSE_i = ln(#visible)."""
    t = rand_head(33, 17, 5)
    res = []
    O, lse = fwd(t["q"], t["k"], t["v"], False, 0.0)
    res += [_close(O, np.tile(t["v"].mean(axis=0), (17, 1)), 1e-13),
            _close(lse, np.full(17, math.log(17)), 1e-13)]
    O, lse = fwd(t["q"], t["k"], t["v"], True, 0.0)
    prefix = np.cumsum(t["v"], axis=0) / np.arange(1, 18)[:, None]
    res += [_close(O, prefix, 1e-13), _close(lse, np.log(np.arange(1, 18)), 1e-13)]
    return _all(res)


def check_causal_first_row(fwd, bwd):
    """Causal row 0 sees key 0 only: O_0 = V_0, LSE_0 = scale q_0.k_0."""
    t = rand_head(34, 40, 8)
    O, lse = fwd(t["q"], t["k"], t["v"], True, 0.35)
    return _all([_close(O[0], t["v"][0], 1e-15),
                 _close(lse[0], 0.35 * t["q"][0] @ t["k"][0], 1e-15)])


# --------------------------------------------------------------------------
# invariants

def check_key_shift(fwd, bwd):
    """k_j -> k_j + u leaves O unchanged and shifts LSE_i by scale q_i.u."""
    res = []
    for causal in (False, True):
        t = rand_head(41, 29, 8)
        u = rand_head(42, 1, 8, ("k",))["k"][0]
        scale = 0.25
        O, lse = fwd(t["q"], t["k"], t["v"], causal, scale)
        O2, lse2 = fwd(t["q"], t["k"] + u, t["v"], causal, scale)
        res += [_close(O2, O, 1e-12), _close(lse2, lse + scale * t["q"] @ u, 1e-12)]
    return _all(res)


def check_permutation(fwd, bwd):
    """Permuting K and V rows jointly leaves non-causal O, LSE unchanged and
    permutes dK, dV the same way."""
    t = rand_head(43, 31, 8)
    perm = np.random.default_rng(7).permutation(31)
    O, lse = fwd(t["q"], t["k"], t["v"], False, 0.3)
    O2, lse2 = fwd(t["q"], t["k"][perm], t["v"][perm], False, 0.3)
    dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], False, 0.3)
    dQ2, dK2, dV2 = bwd(t["q"], t["k"][perm], t["v"][perm], t["do"], False, 0.3)
    return _all([_close(O2, O, 1e-13), _close(lse2, lse, 1e-13), _close(dQ2, dQ, 1e-12),
                 _close(dK2, dK[perm], 1e-12), _close(dV2, dV[perm], 1e-12)])


def check_gradient_sums(fwd, bwd):
    """Rows of dS sum to zero, so sum_j dK_j = 0; rows of P sum to one, so
    sum_j dV_j = sum_i dO_i."""
    res = []
    for causal in (False, True):
        t = rand_head(44, 33, 8)
        dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], causal, 0.3)
        res += [_close(dK.sum(axis=0), np.zeros(8), 1e-12),
                _close(dV.sum(axis=0), t["do"].sum(axis=0), 1e-12)]
    return _all(res)


ALL_CHECKS = (check_golden, check_multiprecision, check_torch_float64,
              check_finite_differences, check_single_token, check_constant_v,
              check_zero_scale, check_causal_first_row, check_key_shift,
              check_permutation, check_gradient_sums)

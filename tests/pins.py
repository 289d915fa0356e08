"""Pin checks for an exact-attention implementation on the CPU.

Each ``check_*`` takes a per-head forward ``fwd(q, k, v, causal, scale)
-> (O, LSE)`` and backward ``bwd(q, k, v, do, causal, scale) -> (dQ, dK, dV)``
(float64 arrays: q and do [Nq, d], k and v [Nk, d]) and returns
``(ok, message)``; the ``check_varlen_*`` ones take the packed-batch
functions described above ``VARLEN_CHECKS``. The oracle tests run
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
    """Rows of q against the rows of k, v; causal rows see keys up to their
    index plus len(k) - len(q) (bottom-right alignment)."""
    import mpmath as mp
    Nq, Nk, d = len(q), len(k), len(q[0])
    O, L = [], []
    for i in range(Nq):
        keys = [j for j in range(Nk) if not (causal and j > i + Nk - Nq)]
        s = {j: scale * mp.fsum(q[i][c] * k[j][c] for c in range(d)) for j in keys}
        z = mp.fsum(mp.exp(s[j]) for j in keys)
        O.append([mp.fsum(mp.exp(s[j]) * v[j][c] for j in keys) / z for c in range(d)])
        L.append(mp.log(z))
    return O, L


def check_multiprecision(fwd, bwd):
    import mpmath as mp
    res = []
    with mp.workdps(40):
        for seed, N, Nk, d, causal in ((1, 1, 1, 2, False), (2, 3, 3, 2, False),
                                       (3, 3, 3, 2, True), (4, 5, 5, 3, True),
                                       (5, 4, 4, 1, False), (6, 2, 4, 2, True),
                                       (7, 3, 2, 2, False), (8, 1, 3, 2, True)):
            t = rand_head(seed, N, d, ("q", "do"))
            t.update(rand_head(seed + 100, Nk, d, ("k", "v")))
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
                rows = N if which == 0 else Nk
                g = np.zeros((rows, d))
                for i in range(rows):
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


# --------------------------------------------------------------------------
# unequal lengths (Nq != Nk): the causal mask is PyTorch's bottom-right
# ("lower right") causal bias, a library definition of the alignment

def _lower_right(nq, nk):
    import warnings
    from torch.nn.attention.bias import causal_lower_right
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        return causal_lower_right(nq, nk)._materialize()


def _torch_reference(q, k, v, do, mask, scale):
    """PyTorch float64 SDPA with a boolean mask (True = visible; None = no
    mask), LSE from torch.logsumexp and gradients from autograd. Every row
    must see at least one key."""
    import torch
    import torch.nn.functional as F
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    out = F.scaled_dot_product_attention(tq[None], tk[None], tv[None], attn_mask=mask,
                                         scale=scale)[0]
    out.backward(torch.tensor(do, dtype=torch.float64))
    s = scale * (tq.detach() @ tk.detach().T)
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    return (out.detach().numpy(), torch.logsumexp(s, dim=1).numpy(), tq.grad.numpy(),
            tk.grad.numpy(), tv.grad.numpy())


def _head_pair(seed, nq, nk, d):
    t = rand_head(seed, nq, d, ("q", "do"))
    t.update(rand_head(seed + 500, nk, d, ("k", "v")))
    return t


def check_torch_unequal(fwd, bwd):
    """Nq != Nk against PyTorch, causal through its lower-right bias. With
    Nq > Nk the first Nq - Nk causal rows see no key; PyTorch is given the
    other rows only, which carry the whole gradient of K and V."""
    res = []
    for seed, nq, nk, d, causal in ((71, 5, 37, 8, True), (72, 1, 50, 8, True),
                                    (73, 20, 70, 4, True), (74, 13, 29, 8, False),
                                    (75, 29, 13, 8, False), (76, 40, 17, 4, True)):
        t = _head_pair(seed, nq, nk, d)
        scale = 1.0 / math.sqrt(d)
        lo = max(nq - nk, 0) if causal else 0
        mask = _lower_right(nq, nk)[lo:] if causal else None
        O_t, lse_t, dq_t, dk_t, dv_t = _torch_reference(t["q"][lo:], t["k"], t["v"],
                                                        t["do"][lo:], mask, scale)
        O, lse = fwd(t["q"], t["k"], t["v"], causal, scale)
        dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], causal, scale)
        res += [_close(O[lo:], O_t, 1e-12), _close(lse[lo:], lse_t, 1e-12),
                _close(dQ[lo:], dq_t, 1e-11), _close(dK, dk_t, 1e-11), _close(dV, dv_t, 1e-11)]
    return _all(res)


def check_suffix_of_square(fwd, bwd):
    """Causal with Nq <= Nk: the result for Q equals the last Nq rows of the
    square causal attention of [X; Q] against the same keys, for any X; with
    dO = 0 on the X rows, the gradients of K and V are those of Q alone."""
    res = []
    for seed, nq, nk in ((81, 7, 19), (82, 1, 12), (83, 12, 12)):
        t = _head_pair(seed, nq, nk, 8)
        x = rand_head(seed + 1, nk - nq, 8, ("q",))["q"]
        qf = np.vstack([x, t["q"]])
        dof = np.vstack([np.zeros((nk - nq, 8)), t["do"]])
        Of, lsef = fwd(qf, t["k"], t["v"], True, 0.3)
        dQf, dKf, dVf = bwd(qf, t["k"], t["v"], dof, True, 0.3)
        O, lse = fwd(t["q"], t["k"], t["v"], True, 0.3)
        dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], True, 0.3)
        res += [_close(O, Of[nk - nq:], 1e-13), _close(lse, lsef[nk - nq:], 1e-13),
                _close(dQ, dQf[nk - nq:], 1e-12), _close(dK, dKf, 1e-12), _close(dV, dVf, 1e-12)]
    return _all(res)


def _neg_inf(x):
    x = np.asarray(x)
    if x.size and np.all(np.isneginf(x)):
        return True, ""
    return False, f"expected -inf, got {x}"


def check_rows_without_keys(fwd, bwd):
    """A query row with no visible key (causal with Nq > Nk, or Nk = 0) has
    O = 0, LSE = -inf and dQ = 0, and the other rows are unaffected by it."""
    res = []
    t = _head_pair(91, 9, 4, 6)
    O, lse = fwd(t["q"], t["k"], t["v"], True, 0.4)
    dQ, dK, dV = bwd(t["q"], t["k"], t["v"], t["do"], True, 0.4)
    O2, lse2 = fwd(t["q"][5:], t["k"], t["v"], True, 0.4)
    dQ2, dK2, dV2 = bwd(t["q"][5:], t["k"], t["v"], t["do"][5:], True, 0.4)
    res += [_close(O[:5], np.zeros((5, 6)), 0.0), _neg_inf(lse[:5]),
            _close(dQ[:5], np.zeros((5, 6)), 0.0), _close(O[5:], O2, 1e-15),
            _close(lse[5:], lse2, 1e-15), _close(dQ[5:], dQ2, 1e-15), _close(dK, dK2, 1e-15),
            _close(dV, dV2, 1e-15)]
    for causal in (False, True):
        e = np.zeros((0, 6))
        O, lse = fwd(t["q"], e, e, causal, 0.4)
        dQ, dK, dV = bwd(t["q"], e, e, t["do"], causal, 0.4)
        res += [_close(O, np.zeros((9, 6)), 0.0), _neg_inf(lse), _close(dQ, np.zeros((9, 6)), 0.0),
                _close(dK, e, 0.0), _close(dV, e, 0.0)]
    return _all(res)


ALL_CHECKS = (check_golden, check_multiprecision, check_torch_float64,
              check_finite_differences, check_single_token, check_constant_v,
              check_zero_scale, check_causal_first_row, check_key_shift,
              check_permutation, check_gradient_sums, check_torch_unequal,
              check_suffix_of_square, check_rows_without_keys)


# --------------------------------------------------------------------------
# packed batches: ``vfwd(q, k, v, cu_q, cu_k, causal, scale) -> (O [Tq,H,d],
# LSE [H,Tq])`` and ``vbwd(q, k, v, do, cu_q, cu_k, causal, scale) -> (dQ, dK,
# dV)`` over q [Tq, H, d], k, v [Tk, H, d]

def packed_inputs(seed, lens_q, lens_k, H, d):
    """Packed [T, H, d] tensors whose (sequence b, head h) block is the seeded
    head generator's output for (b, h), and the prefix offsets."""
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int64)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int64)
    x = {"q": np.zeros((cu_q[-1], H, d)), "do": np.zeros((cu_q[-1], H, d)),
         "k": np.zeros((cu_k[-1], H, d)), "v": np.zeros((cu_k[-1], H, d))}
    for b, (nq, nk) in enumerate(zip(lens_q, lens_k)):
        for h in range(H):
            tq = rand_head(seed, nq, d, ("q", "do"), b=b, h=h)
            tk = rand_head(seed + 500, nk, d, ("k", "v"), b=b, h=h)
            for n, t, c in (("q", tq, cu_q), ("do", tq, cu_q), ("k", tk, cu_k), ("v", tk, cu_k)):
                x[n][c[b]:c[b + 1], h] = t[n]
    return x, cu_q, cu_k


def check_varlen_block_diagonal(vfwd, vbwd):
    """A packed batch equals PyTorch's attention over the whole packed token
    axis with a block-diagonal mask: token rows of one sequence see only that
    sequence's keys, causally through PyTorch's lower-right bias. Lengths
    differ between sequences and include an empty one."""
    import torch
    res = []
    lens_q, lens_k = [5, 0, 17, 1, 9, 3], [7, 3, 17, 12, 9, 3]
    x, cu_q, cu_k = packed_inputs(101, lens_q, lens_k, 2, 4)
    for causal in (False, True):
        mask = torch.zeros(cu_q[-1], cu_k[-1], dtype=torch.bool)
        for b in range(len(lens_q)):
            blk = _lower_right(lens_q[b], lens_k[b]) if causal else True
            mask[cu_q[b]:cu_q[b + 1], cu_k[b]:cu_k[b + 1]] = blk
        O, lse = vfwd(x["q"], x["k"], x["v"], cu_q, cu_k, causal, 0.45)
        dQ, dK, dV = vbwd(x["q"], x["k"], x["v"], x["do"], cu_q, cu_k, causal, 0.45)
        for h in range(2):
            O_t, lse_t, dq_t, dk_t, dv_t = _torch_reference(
                x["q"][:, h], x["k"][:, h], x["v"][:, h], x["do"][:, h], mask, 0.45)
            res += [_close(O[:, h], O_t, 1e-12), _close(lse[h], lse_t, 1e-12),
                    _close(dQ[:, h], dq_t, 1e-11), _close(dK[:, h], dk_t, 1e-11),
                    _close(dV[:, h], dv_t, 1e-11)]
    return _all(res)


def check_varlen_rows_without_keys(vfwd, vbwd):
    """Sequence 0 has no keys: O = 0, LSE = -inf, dQ = 0. Sequence 1 has 3
    queries and 2 keys, causal: its first query sees nothing, its second sees
    key 0 only (O = V_0, LSE = scale q.k_0), its third sees both keys."""
    res = []
    x, cu_q, cu_k = packed_inputs(111, [4, 3], [0, 2], 1, 4)
    O, lse = vfwd(x["q"], x["k"], x["v"], cu_q, cu_k, True, 0.6)
    dQ, dK, dV = vbwd(x["q"], x["k"], x["v"], x["do"], cu_q, cu_k, True, 0.6)
    q, k, v = x["q"][:, 0], x["k"][:, 0], x["v"][:, 0]
    res += [_close(O[:5, 0], np.zeros((5, 4)), 0.0), _neg_inf(lse[0, :5]),
            _close(dQ[:5, 0], np.zeros((5, 4)), 0.0), _close(O[5, 0], v[0], 1e-15),
            _close(lse[0, 5], 0.6 * q[5] @ k[0], 1e-15)]
    O_t, lse_t, _, _, _ = _torch_reference(q[6:], k, v, x["do"][6:, 0], None, 0.6)
    res += [_close(O[6:, 0], O_t, 1e-12), _close(lse[0, 6:], lse_t, 1e-12)]
    return _all(res)


VARLEN_CHECKS = (check_varlen_block_diagonal, check_varlen_rows_without_keys)

"""Plants plausible mistakes in copies of the oracle and requires the pin
checks to catch every one. This shows that the pins would catch such a slip
in the oracle itself. CPU only.
"""

import numpy as np
import pytest

from oracle import attention as orc

from . import pins

pytest.importorskip("mpmath")
pytest.importorskip("torch")


def _scores(q, k, causal, scale, mask_shift=0, mask_dir=1, use_scale=True, align=1):
    nq, nk = q.shape[0], k.shape[0]
    S = (scale if use_scale else 1.0) * (q @ k.T)
    if causal:
        i = np.arange(nq)[:, None] + align * (nk - nq)
        j = np.arange(nk)[None, :]
        masked = (mask_dir * (j - i)) > -mask_shift
        S = np.where(masked, -np.inf, S)
    return S


def _softmax(S, log=np.log):
    if S.shape[1] == 0:
        return np.zeros(S.shape), np.full(S.shape[0], -np.inf)
    m = S.max(axis=1)
    empty = ~np.isfinite(m)
    m = np.where(empty, 0.0, m)
    E = np.exp(S - m[:, None])
    l = np.where(empty, 1.0, E.sum(axis=1))
    with np.errstate(divide="ignore"):
        return E / l[:, None], np.where(empty, -np.inf, m + log(l))


def make_fwd(**kw):
    log = kw.pop("log", np.log)
    transpose_p = kw.pop("transpose_p", False)

    def fwd(q, k, v, causal, scale):
        P, lse = _softmax(_scores(q, k, causal, scale, **kw), log)
        return ((P.T if transpose_p else P) @ v), lse
    return fwd


def make_bwd(drop_d=False, dk_scale=True, dq_transposed=False, dv_untransposed=False,
             sign=1.0):
    def bwd(q, k, v, do, causal, scale):
        P, _ = _softmax(_scores(q, k, causal, scale))
        if dq_transposed and P.shape[0] != P.shape[1]:
            raise ValueError("dS^T K needs a square dS")
        dV = (P if dv_untransposed else P.T) @ do
        dP = do @ v.T
        D = (P * dP).sum(axis=1)
        dS = P * (dP - (0.0 if drop_d else D[:, None])) * sign
        dQ = scale * ((dS.T if dq_transposed else dS) @ k)
        dK = (scale if dk_scale else 1.0) * (dS.T @ q)
        return dQ, dK, dV
    return bwd


GOOD_FWD = make_fwd()
GOOD_BWD = make_bwd()

MUTANTS = {
    "scale dropped from the scores": (make_fwd(use_scale=False), GOOD_BWD),
    "causal mask off by one (diagonal masked)": (make_fwd(mask_shift=1), GOOD_BWD),
    "causal mask in the wrong direction": (make_fwd(mask_dir=-1), GOOD_BWD),
    "P transposed in O = P V": (make_fwd(transpose_p=True), GOOD_BWD),
    "log2 instead of ln in the LSE": (make_fwd(log=np.log2), GOOD_BWD),
    "D dropped from dS": (GOOD_FWD, make_bwd(drop_d=True)),
    "scale dropped from dK": (GOOD_FWD, make_bwd(dk_scale=False)),
    "dS transposed in dQ": (GOOD_FWD, make_bwd(dq_transposed=True)),
    "P not transposed in dV": (GOOD_FWD, make_bwd(dv_untransposed=True)),
    "sign of dS flipped": (GOOD_FWD, make_bwd(sign=-1.0)),
    "top-left causal alignment when Nq != Nk": (make_fwd(align=0), GOOD_BWD),
    "bottom-right offset with the wrong sign": (make_fwd(align=-1), GOOD_BWD),
}

# The checks are run cheapest first; a mutant is caught at its first failure.
ORDER = (pins.check_single_token, pins.check_causal_first_row, pins.check_zero_scale,
         pins.check_golden, pins.check_gradient_sums, pins.check_key_shift,
         pins.check_permutation, pins.check_constant_v, pins.check_torch_float64,
         pins.check_finite_differences, pins.check_rows_without_keys,
         pins.check_suffix_of_square, pins.check_torch_unequal)


def caught(fwd, bwd):
    import warnings
    for check in ORDER:
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            try:
                ok, _ = check(fwd, bwd)
            except (FloatingPointError, ValueError):
                ok = False
        if not ok:
            return check.__name__
    return None


def test_unmutated_copy_passes():
    assert caught(GOOD_FWD, GOOD_BWD) is None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    fwd, bwd = MUTANTS[name]
    assert caught(fwd, bwd) is not None, f"no pin catches: {name}"


def test_oracle_module_is_what_the_copy_mirrors():
    """The unmutated copy and the oracle agree, so the mutants are mutations
    of the oracle's arithmetic."""
    t = pins.rand_head(99, 21, 8)
    for causal in (False, True):
        a = GOOD_FWD(t["q"], t["k"], t["v"], causal, 0.3)
        b = orc.head_forward(t["q"], t["k"], t["v"], causal, 0.3)
        assert np.max(np.abs(a[0] - b[0])) < 1e-13 and np.max(np.abs(a[1] - b[1])) < 1e-13
        ga = GOOD_BWD(t["q"], t["k"], t["v"], t["do"], causal, 0.3)
        gb = orc.head_backward(t["q"], t["k"], t["v"], t["do"], causal, 0.3)
        for x, y in zip(ga, gb):
            assert np.max(np.abs(x - y)) < 1e-12
    for nq, nk in ((7, 19), (19, 7)):
        t = pins._head_pair(98, nq, nk, 8)
        a = GOOD_FWD(t["q"], t["k"], t["v"], True, 0.3)
        b = orc.head_forward(t["q"], t["k"], t["v"], True, 0.3)
        assert np.array_equal(np.isneginf(a[1]), np.isneginf(b[1]))
        fin = np.isfinite(b[1])
        assert np.max(np.abs(a[0] - b[0])) < 1e-13 and np.max(np.abs(a[1][fin] - b[1][fin])) < 1e-13


# --------------------------------------------------------------------------
# packed batches: a copy of the oracle's per-sequence loop with planted slips

def make_vfwd(slip=None):
    def vfwd(q, k, v, cu_q, cu_k, causal, scale):
        Tq, H, d = q.shape
        O = np.zeros((Tq, H, d))
        lse = np.empty((H, Tq))
        for b in range(len(cu_q) - 1):
            q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
            if slip == "keys sliced with the query offsets":
                k0, k1 = q0, q0 + (k1 - k0)
            if slip == "key block of the next sequence" and b + 2 < len(cu_k):
                k0, k1 = cu_k[b + 1], cu_k[b + 1] + (k1 - k0)
            for h in range(H):
                kk, vv = k[k0:k1, h], v[k0:k1, h]
                if slip == "heads of K swapped" and H > 1:
                    kk = k[k0:k1, H - 1 - h]
                o, l_ = GOOD_FWD(q[q0:q1, h], kk, vv, causal, scale)
                O[q0:q1, h], lse[h, q0:q1] = o, l_
        return O, lse
    return vfwd


def make_vbwd():
    def vbwd(q, k, v, do, cu_q, cu_k, causal, scale):
        dQ, dK, dV = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
        for b in range(len(cu_q) - 1):
            q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
            for h in range(q.shape[1]):
                dQ[q0:q1, h], dK[k0:k1, h], dV[k0:k1, h] = GOOD_BWD(
                    q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], do[q0:q1, h], causal, scale)
        return dQ, dK, dV
    return vbwd


VARLEN_MUTANTS = ("keys sliced with the query offsets", "key block of the next sequence",
                  "heads of K swapped")


def vcaught(vfwd, vbwd):
    import warnings
    for check in pins.VARLEN_CHECKS:
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            try:
                ok, _ = check(vfwd, vbwd)
            except (FloatingPointError, ValueError, IndexError):
                ok = False
        if not ok:
            return check.__name__
    return None


def test_unmutated_varlen_copy_passes():
    assert vcaught(make_vfwd(), make_vbwd()) is None


@pytest.mark.parametrize("name", VARLEN_MUTANTS)
def test_varlen_mutant_is_caught(name):
    assert vcaught(make_vfwd(name), make_vbwd()) is not None, f"no pin catches: {name}"

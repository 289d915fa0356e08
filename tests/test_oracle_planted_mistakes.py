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


def _scores(q, k, causal, scale, mask_shift=0, mask_dir=1, use_scale=True):
    N = k.shape[0]
    S = (scale if use_scale else 1.0) * (q @ k.T)
    if causal:
        i = np.arange(N)[:, None]
        j = np.arange(N)[None, :]
        masked = (mask_dir * (j - i)) > -mask_shift
        S = np.where(masked, -np.inf, S)
    return S


def _softmax(S, log=np.log):
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])
    l = E.sum(axis=1)
    return E / l[:, None], m + log(l)


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
}

# The checks are run cheapest first; a mutant is caught at its first failure.
ORDER = (pins.check_single_token, pins.check_causal_first_row, pins.check_zero_scale,
         pins.check_golden, pins.check_gradient_sums, pins.check_key_shift,
         pins.check_permutation, pins.check_constant_v, pins.check_torch_float64,
         pins.check_finite_differences)


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

"""Backward parity: the CUDA backward through the C ABI against the fp64 oracle.

The backward consumes the forward's own O and LSE (as a training step does);
the oracle computes its gradients from the inputs alone.
"""

import numpy as np
import pytest

import oracle

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _grads(fa, dev, causal, scale):
    o, lse = gu.run_fwd(fa, dev, causal, scale)
    return [gu.to_f64(g) for g in gu.run_bwd(fa, dev, o, lse, causal, scale)]


def _full_check(fa, seed, B, H, N, d, causal, scale=None):
    scale = gu.default_scale(d) if scale is None else scale
    dev, bits = gu.device_inputs(seed, B, H, N, d)
    got = _grads(fa, dev, causal, scale)
    x = {n: np.stack([np.stack([gu.head_f64(bits, b, h, (n,))[n] for h in range(H)])
                      for b in range(B)]) for n in ("q", "k", "v", "do")}
    want = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
    gu.check_grads(got, want, f"B={B} H={H} N={N} d={d} causal={causal}")
    return got, x


@pytest.mark.parametrize("causal", [False, True])
def test_config_b4_h8_n1024_d64(cuda_lib, causal):
    _full_check(cuda_lib, 2, 4, 8, 1024, 64, causal)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 77, 128, 129, 200, 383, 640])
def test_ragged_lengths(cuda_lib, N, d, causal):
    _full_check(cuda_lib, 100 + N, 2, 3, N, d, causal)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_heads_spread_over_persistent_ctas(cuda_lib, d, causal):
    _full_check(cuda_lib, 8, 3, 40, 384, d, causal)


@pytest.mark.parametrize("scale", [0.0, 0.5])
def test_other_scales(cuda_lib, scale):
    _full_check(cuda_lib, 9, 1, 2, 300, 64, True, scale)
    _full_check(cuda_lib, 9, 1, 2, 300, 128, False, scale)


def test_single_token_closed_form(cuda_lib):
    """N = 1: P = 1, so dV = dO exactly and dS = dP - D = 0 up to the fp32
    rounding of two dot products summed in different orders."""
    dev, bits = gu.device_inputs(10, 2, 2, 1, 64)
    dq, dk, dv = _grads(cuda_lib, dev, True, 0.125)
    assert np.max(np.abs(dq)) < 1e-4 and np.max(np.abs(dk)) < 1e-4
    assert np.array_equal(dv, gu.to_f64(dev["do"]))


def test_repeated_calls_are_independent(cuda_lib):
    """The workspace is re-initialised by every call: two calls give the same
    gradients bit for bit."""
    dev, _ = gu.device_inputs(11, 1, 4, 500, 128)
    o, lse = gu.run_fwd(cuda_lib, dev, True, 0.1)
    g1 = [gu.to_f64(g) for g in gu.run_bwd(cuda_lib, dev, o, lse, True, 0.1)]
    g2 = [gu.to_f64(g) for g in gu.run_bwd(cuda_lib, dev, o, lse, True, 0.1)]
    for a, b in zip(g1[1:], g2[1:]):  # dK, dV are computed without atomics
        assert np.array_equal(a, b)
    assert gu.rel_l2(g1[0], g2[0]) < 1e-2  # dQ: fp32 atomics, order may vary


# ---------------------------------------------------------------------------
# full sizes: gradient-sum invariants on every head, the oracle on sampled heads

def _invariants(dk, dv, do, what):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i for every (b, h)."""
    sdo = do.sum(axis=2)
    err_v = np.abs(dv.sum(axis=2) - sdo) / (np.abs(sdo) + np.sqrt(do.shape[2]))
    assert err_v.max() < 2e-2, f"{what}: sum dV vs sum dO {err_v.max():.3e}"
    scale_k = np.sqrt((dk ** 2).sum(axis=2))
    err_k = np.abs(dk.sum(axis=2)) / (scale_k + 1e-30)
    assert err_k.max() < 5e-2, f"{what}: sum dK {err_k.max():.3e}"


SWEEP = [(d, H, N) for d, H in ((64, 32), (128, 16))
         for N in (512, 1024, 2048, 4096, 8192, 16384)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,H,N", SWEEP)
def test_gpt_sweep_full_size(cuda_lib, d, H, N, causal):
    B = 16384 // N
    scale = gu.default_scale(d)
    dev, bits = gu.device_inputs(30 + N + d, B, H, N, d)
    dq, dk, dv = _grads(cuda_lib, dev, causal, scale)
    what = f"N={N} d={d} causal={causal}"
    for g in (dq, dk, dv):
        assert np.all(np.isfinite(g)), what
    _invariants(dk, dv, gu.to_f64(dev["do"]), what)
    heads = gu.sample_heads(B, H, 2 if N <= 4096 else 1, seed=N + d)
    for b, h in heads:
        x = gu.head_f64(bits, b, h)
        want = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
        gu.check_grads((dq[b, h], dk[b, h], dv[b, h]), want, f"{what} head ({b},{h})")


def test_long_sequence_causal_full_size(cuda_lib):
    """B=1, H=16, N=32768, d=128, causal: invariants on all heads, the oracle on
    the last head, sampled dQ rows on two more."""
    B, H, N, d = 1, 16, 32768, 128
    scale = gu.default_scale(d)
    dev, bits = gu.device_inputs(50, B, H, N, d)
    dq, dk, dv = _grads(cuda_lib, dev, True, scale)
    _invariants(dk, dv, gu.to_f64(dev["do"]), "N=32768")
    x = gu.head_f64(bits, 0, H - 1)
    want = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], True, scale)
    gu.check_grads((dq[0, H - 1], dk[0, H - 1], dv[0, H - 1]), want, "N=32768 last head")
    rows = gu.sample_rows(N, seed=3)
    for h in (0, 7):
        x = gu.head_f64(bits, 0, h)
        dq_rows, _, _ = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], True, scale,
                                             rows=rows)
        rl = gu.rel_l2(dq[0, h, rows], dq_rows)
        assert rl <= gu.TOL_GRAD_RELL2, f"head {h}: sampled dQ rows rel-L2 {rl:.3e}"

"""Backward parity at head dimension 256 (its own dK / dV kernel over 64-key
blocks, with dK^T, dV^T and dQ^T in TMEM by head-dim halves) through the C
ABI against the fp64 oracle. The backward consumes the forward's O and LSE."""

import numpy as np
import pytest

import oracle

from . import gpu_util as gu
from .test_bwd_gpu import _full_check, _grads, _invariants

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 77, 128, 129, 192, 200, 256, 383, 640])
def test_d256_bwd_ragged_lengths(cuda_lib, N, causal):
    """Lengths around the 64-key and 128-query block edges, where the causal
    diagonal of an odd key block starts half way down a query block."""
    _full_check(cuda_lib, 700 + N, 2, 3, N, 256, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_d256_bwd_many_heads_spread_over_persistent_ctas(cuda_lib, causal):
    """Many more items than SMs: every CTA hands its dK^T / dV^T columns from
    one item's epilogue to the next item's first MMAs, and its Q / dO buffer
    from block to block."""
    _full_check(cuda_lib, 710, 3, 40, 384, 256, causal)


@pytest.mark.parametrize("scale", [0.0, 0.5])
def test_d256_bwd_other_scales(cuda_lib, scale):
    _full_check(cuda_lib, 711, 1, 2, 300, 256, True, scale)
    _full_check(cuda_lib, 711, 1, 2, 300, 256, False, scale)


def test_d256_bwd_single_token_closed_form(cuda_lib):
    """N = 1: P = 1, so dV = dO exactly and dS = dP - D = 0 up to rounding."""
    dev, _ = gu.device_inputs(712, 2, 2, 1, 256)
    dq, dk, dv = _grads(cuda_lib, dev, True, 0.0625)
    assert np.max(np.abs(dq)) < 1e-4 and np.max(np.abs(dk)) < 1e-4
    assert np.array_equal(dv, gu.to_f64(dev["do"]))


def test_d256_bwd_repeated_calls(cuda_lib):
    """dK and dV are written without atomics: two calls agree bit for bit."""
    dev, _ = gu.device_inputs(713, 1, 4, 500, 256)
    o, lse = gu.run_fwd(cuda_lib, dev, True, 0.1)
    g1 = [gu.to_f64(g) for g in gu.run_bwd(cuda_lib, dev, o, lse, True, 0.1)]
    g2 = [gu.to_f64(g) for g in gu.run_bwd(cuda_lib, dev, o, lse, True, 0.1)]
    for a, b in zip(g1[1:], g2[1:]):
        assert np.array_equal(a, b)
    assert gu.rel_l2(g1[0], g2[0]) < 1e-2


def test_d256_bwd_strided_layout(cuda_lib):
    """[B, N, H, d] storage passed as [B, H, N, d] views for every tensor
    gives the same bits as the contiguous call."""
    import torch
    fa = cuda_lib
    B, H, N, d = 2, 3, 300, 256
    dev, _ = gu.device_inputs(714, B, H, N, d)
    for causal in (False, True):
        o, lse = gu.run_fwd(fa, dev, causal, 0.0625)
        ref = gu.run_bwd(fa, dev, o, lse, causal, 0.0625)
        v = {n: t.transpose(1, 2).contiguous().transpose(1, 2) for n, t in dev.items()}
        ov = o.transpose(1, 2).contiguous().transpose(1, 2)
        grads = [torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
                 for _ in range(3)]
        ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
        fa.fa_bwd(v["q"], v["k"], v["v"], ov, lse, v["do"], *grads, causal, 0.0625, ws)
        assert fa.fa_last_device_status() == fa.FA_OK
        for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
            if name == "dQ":  # fp32 atomics: the order of the additions may differ
                assert gu.rel_l2(gu.to_f64(g), gu.to_f64(r)) < 1e-2
            else:
                assert torch.equal(g, r), name


@pytest.mark.parametrize("causal", [False, True])
def test_d256_bwd_full_size_sampled(cuda_lib, causal):
    """B = 2, H = 16, N = 4096 (the d = 256 bench shape): gradient-sum
    invariants on every head, the oracle on two sampled heads."""
    B, H, N, d = 2, 16, 4096, 256
    scale = gu.default_scale(d)
    dev, bits = gu.device_inputs(715, B, H, N, d)
    dq, dk, dv = _grads(cuda_lib, dev, causal, scale)
    what = f"N={N} d={d} causal={causal}"
    for g in (dq, dk, dv):
        assert np.all(np.isfinite(g)), what
    _invariants(dk, dv, gu.to_f64(dev["do"]), what)
    for b, h in gu.sample_heads(B, H, 2, seed=716):
        x = gu.head_f64(bits, b, h)
        want = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
        gu.check_grads((dq[b, h], dk[b, h], dv[b, h]), want, f"{what} head ({b},{h})")

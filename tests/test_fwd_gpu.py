"""Forward parity: the CUDA forward through the C ABI against the fp64 oracle."""

import numpy as np
import pytest

import oracle

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _full_check(fa, seed, B, H, N, d, causal, scale=None):
    raw = scale is None or scale == gu.default_scale(d)  # the configs' scale: raw O bound
    scale = gu.default_scale(d) if scale is None else scale
    dev, bits = gu.device_inputs(seed, B, H, N, d, ("q", "k", "v"))
    o, lse = gu.run_fwd(fa, dev, causal, scale)
    og, lg = gu.to_f64(o), gu.to_f64(lse)
    x = {n: np.stack([np.stack([gu.head_f64(bits, b, h, (n,))[n] for h in range(H)])
                      for b in range(B)]) for n in ("q", "k", "v")}
    ow, lw = oracle.attention_forward(x["q"], x["k"], x["v"], causal, scale)
    return gu.check_o_lse(og, lg, ow, lw, f"B={B} H={H} N={N} d={d} causal={causal}", raw=raw)


def test_config_small_noncausal(cuda_lib):
    """B=1, H=2, N=128, d=64, non-causal, scale 1/sqrt(64)."""
    _full_check(cuda_lib, 1, 1, 2, 128, 64, False)


@pytest.mark.parametrize("causal", [False, True])
def test_config_b4_h8_n1024_d64(cuda_lib, causal):
    _full_check(cuda_lib, 2, 4, 8, 1024, 64, causal)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 77, 128, 129, 200, 256, 383, 640])
def test_ragged_lengths(cuda_lib, N, d, causal):
    """Any N >= 1: partial key tiles, partial query tiles, an odd number of
    query tiles (a work item with one live tile), single rows."""
    _full_check(cuda_lib, 3 + N, 2, 3, N, d, causal)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_heads_spread_over_persistent_ctas(cuda_lib, d, causal):
    """More work items than SMs, so every CTA takes several items in turn."""
    _full_check(cuda_lib, 5, 3, 40, 384, d, causal)


@pytest.mark.parametrize("scale", [0.0, 0.05, 0.5])
def test_other_scales(cuda_lib, scale):
    """scale = 0 gives the (prefix) mean of V; large scales give peaked rows."""
    _full_check(cuda_lib, 6, 1, 2, 300, 64, True, scale)
    _full_check(cuda_lib, 6, 1, 2, 300, 128, False, scale)


def test_constant_rows_give_exact_mean(cuda_lib):
    """Equal keys: every visible key has the same weight, O is the mean of V."""
    import torch
    B, H, N, d = 1, 2, 256, 64
    dev, bits = gu.device_inputs(7, B, H, N, d, ("q", "k", "v"))
    k = dev["k"].clone()
    k[:] = k[:, :, :1, :]
    o = torch.empty_like(dev["q"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    cuda_lib.fa_fwd(dev["q"], k, dev["v"], o, lse, False, 0.125)
    v = gu.to_f64(dev["v"])
    og = gu.to_f64(o)
    want = np.broadcast_to(v.mean(axis=2, keepdims=True), og.shape)
    assert gu.max_abs(og, want) < 1e-2


# ---------------------------------------------------------------------------
# the GPT-style sweeps and the long-sequence case at full size, checked on
# sampled heads (always including the last one) and sampled rows

SWEEP = [(d, H, N) for d, H in ((64, 32), (128, 16))
         for N in (512, 1024, 2048, 4096, 8192, 16384)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,H,N", SWEEP)
def test_gpt_sweep_full_size(cuda_lib, d, H, N, causal):
    B = 16384 // N
    scale = gu.default_scale(d)
    dev, bits = gu.device_inputs(30 + N + d, B, H, N, d, ("q", "k", "v"))
    o, lse = gu.run_fwd(cuda_lib, dev, causal, scale)
    og, lg = gu.to_f64(o), gu.to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    rows = gu.sample_rows(N, seed=N)
    for b, h in gu.sample_heads(B, H, 2, seed=N + d):
        x = gu.head_f64(bits, b, h, ("q", "k", "v"))
        ow, lw = oracle.head_forward(x["q"], x["k"], x["v"], causal, scale, rows=rows)
        gu.check_o_lse(og[b, h, rows], lg[b, h, rows], ow, lw, f"head ({b},{h}) N={N} d={d}")


def test_long_sequence_causal_full_size(cuda_lib):
    """B=1, H=16, N=32768, d=128, causal: four heads, sampled rows."""
    B, H, N, d = 1, 16, 32768, 128
    scale = gu.default_scale(d)
    dev, bits = gu.device_inputs(50, B, H, N, d, ("q", "k", "v"))
    o, lse = gu.run_fwd(cuda_lib, dev, True, scale)
    og, lg = gu.to_f64(o), gu.to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    rows = gu.sample_rows(N, seed=5)
    for b, h in gu.sample_heads(B, H, 4, seed=9):
        x = gu.head_f64(bits, b, h, ("q", "k", "v"))
        ow, lw = oracle.head_forward(x["q"], x["k"], x["v"], True, scale, rows=rows)
        gu.check_o_lse(og[b, h, rows], lg[b, h, rows], ow, lw, f"head ({b},{h})")

"""Forward parity at head dimension 256 (its own kernel: one query tile per
CTA with a double-buffered S in TMEM) through the C ABI against the fp64
oracle. The backward at d = 256 is covered in test_bwd256_gpu.py."""

import numpy as np
import pytest

import oracle

from . import gpu_util as gu
from .test_fwd_gpu import _full_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 77, 128, 129, 200, 256, 383, 640])
def test_d256_ragged_lengths(cuda_lib, N, causal):
    _full_check(cuda_lib, 600 + N, 2, 3, N, 256, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_d256_many_heads_spread_over_persistent_ctas(cuda_lib, causal):
    """Many more items than SMs: every CTA reloads Q and reuses its TMEM O for
    several items in turn (the o_free hand-off between items)."""
    _full_check(cuda_lib, 610, 3, 40, 384, 256, causal)


@pytest.mark.parametrize("scale", [0.0, 0.5])
def test_d256_other_scales(cuda_lib, scale):
    _full_check(cuda_lib, 611, 1, 2, 300, 256, True, scale)


def test_d256_strided_layout(cuda_lib):
    """[B, N, H, d] storage passed as [B, H, N, d] views."""
    import torch
    fa = cuda_lib
    B, H, N, d = 2, 3, 300, 256
    dev, bits = gu.device_inputs(612, B, H, N, d, ("q", "k", "v"))
    for causal in (False, True):
        o_ref, l_ref = gu.run_fwd(fa, dev, causal, 0.0625)
        v = {n: t.transpose(1, 2).contiguous().transpose(1, 2) for n, t in dev.items()}
        o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        fa.fa_fwd(v["q"], v["k"], v["v"], o, lse, causal, 0.0625)
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_d256_full_size_sampled(cuda_lib, causal):
    """B = 2, H = 16, N = 4096: sampled heads and rows against the oracle."""
    fa = cuda_lib
    B, H, N, d = 2, 16, 4096, 256
    scale = gu.default_scale(d)
    dev, bits = gu.device_inputs(613, B, H, N, d, ("q", "k", "v"))
    o, lse = gu.run_fwd(fa, dev, causal, scale)
    og, lg = gu.to_f64(o), gu.to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    rows = gu.sample_rows(N, seed=1, n_mid=64)
    for b, h in gu.sample_heads(B, H, 3, seed=2):
        x = gu.head_f64(bits, b, h, ("q", "k", "v"))
        ow, lw = oracle.head_forward(x["q"], x["k"], x["v"], causal, scale, rows=rows)
        gu.check_o_lse(og[b, h, rows], lg[b, h, rows], ow, lw, f"b={b} h={h}")

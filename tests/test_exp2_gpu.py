"""The forward softmax's FMA-pipe exponential, evaluated on the device through
the C ABI, against float64 2^x: relative error below 1e-4 on the range the
softmax uses (x in [-125, 8]; 8 is the deferred-rescale threshold)."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_exp2_polynomial_error_bound(cuda_lib):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.uniform(-125.0, 8.0, 1_000_000),
        np.arange(-125.0, 8.0, 0.125),            # integers, halves, ties of the rounding
        [0.0, -0.0, 0.5, -0.5, 1e-7, -1e-7, 7.999, -124.999],
    ]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty_like(xd)
    cuda_lib.fa_selftest_exp2(xd, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1e-4, f"max relative error {rel.max():.3e} at x={x[np.argmax(rel)]}"


def test_exp2_polynomial_clamps_below_minus_125(cuda_lib):
    """Below -125 the value stays the normal number 2^-125 (callers zero masked
    entries themselves)."""
    x = torch.tensor([-126.0, -200.0, float("-inf")], device="cuda")
    y = torch.empty_like(x)
    cuda_lib.fa_selftest_exp2(x, y)
    torch.cuda.synchronize()
    ref = 2.0 ** -125
    assert np.allclose(y.cpu().numpy(), ref, rtol=1e-4)

"""The two dQ paths of the backward, through fa_bwd_with_dq_path, against the
fp64 oracle: FA_DQ_ATOMIC (the dK/dV kernel adds dS K per tile with atomics)
and FA_DQ_SEPARATE (the dK/dV kernel without dQ, then a query-stationary
kernel that sums dQ in tensor memory). The separate path gives the same dq
bits on every run."""

import numpy as np
import pytest

import oracle

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _bwd(fa, dev, o, lse, causal, scale, dq_path):
    import torch
    q = dev["q"]
    B, H, N, d = q.shape
    ws = torch.full((fa.fa_bwd_workspace_size(B, H, N, d),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.fa_bwd(q, dev["k"], dev["v"], o, lse, dev["do"], *grads, causal, scale, ws,
              dq_path=dq_path)
    assert fa.fa_last_device_status() == fa.FA_OK
    return [gu.to_f64(g) for g in grads]


def _check(fa, seed, B, H, N, d, causal, heads=None, scale=None):
    scale = gu.default_scale(d) if scale is None else scale
    dev, bits = gu.device_inputs(seed, B, H, N, d)
    o, lse = gu.run_fwd(fa, dev, causal, scale)
    sep = _bwd(fa, dev, o, lse, causal, scale, fa.FA_DQ_SEPARATE)
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in heads:
        x = gu.head_f64(bits, b, h)
        want = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
        gu.check_grads([g[b, h] for g in sep], want,
                       f"separate dQ path B={B} H={H} N={N} d={d} causal={causal} ({b},{h})")
    return dev, o, lse, sep, scale


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 77, 128, 129, 383, 640])
def test_separate_dq_ragged_lengths(cuda_lib, N, d, causal):
    _check(cuda_lib, 700 + N, 2, 3, N, d, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_separate_dq_many_items_per_cta(cuda_lib, d, causal):
    """More query blocks than SMs: every CTA takes several items in turn, and
    items of different lengths follow each other (causal)."""
    _check(cuda_lib, 710, 2, 40, 1024, d, causal, heads=gu.sample_heads(2, 40, 3, seed=d))


@pytest.mark.parametrize("causal", [False, True])
def test_separate_dq_long_sequence_sampled(cuda_lib, causal):
    """Config-4 size (B = 4, H = 16, N = 4096, d = 128) on two sampled heads."""
    _check(cuda_lib, 720, 4, 16, 4096, 128, causal, heads=[(0, 3), (3, 15)])


def test_separate_dq_is_bitwise_reproducible_and_agrees_with_atomic(cuda_lib):
    fa = cuda_lib
    dev, o, lse, sep, scale = _check(fa, 730, 2, 8, 1000, 128, True, heads=[(1, 7)])
    again = _bwd(fa, dev, o, lse, True, scale, fa.FA_DQ_SEPARATE)
    for a, b in zip(sep, again):
        assert np.array_equal(a, b)
    atomic = _bwd(fa, dev, o, lse, True, scale, fa.FA_DQ_ATOMIC)
    for name, a, b in zip(("dQ", "dK", "dV"), sep, atomic):
        assert gu.rel_l2(a, b) < 1e-2, name


def test_dq_path_arguments(cuda_lib):
    import torch
    fa = cuda_lib
    dev, _ = gu.device_inputs(740, 1, 2, 256, 96)
    o, lse = gu.run_fwd(fa, dev, False, 0.1)
    ws = torch.empty(fa.fa_bwd_workspace_size(1, 2, 256, 96), dtype=torch.uint8, device="cuda")
    g = [torch.empty_like(dev["q"]) for _ in range(3)]
    with pytest.raises(fa.FaError) as e:  # the separate kernel takes d = 64 and 128
        fa.fa_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], *g, False, 0.1, ws,
                  dq_path=fa.FA_DQ_SEPARATE)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], *g, False, 0.1, ws, dq_path=7)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    for path in (fa.FA_DQ_AUTO, fa.FA_DQ_ATOMIC):  # every d takes these
        fa.fa_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], *g, False, 0.1, ws,
                  dq_path=path)
    assert fa.fa_last_device_status() == fa.FA_OK

"""Strided layouts through fa_fwd_strided / fa_bwd_strided: [B, N, H, d]
tensors (as flash_attn_func takes them) and K/V packed in one [B, N, 2, H, d]
buffer give the same results as the contiguous [B, H, N, d] call: O, LSE, dK
and dV bit for bit (same kernels, same arithmetic), dQ within the atomics'
rounding-order tolerance; and one ragged case against the oracle."""

import numpy as np
import pytest
import torch

import oracle

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _run(fa, q, k, v, do, o, lse, dq, dk, dv, causal, scale):
    fa.fa_fwd(q, k, v, o, lse, causal, scale)
    B, H, N, d = q.shape
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal, scale, ws)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK


def _contiguous_reference(fa, dev, causal, scale):
    q = dev["q"]
    out = [torch.empty_like(q)] + [torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")] + \
          [torch.empty_like(q) for _ in range(3)]
    _run(fa, dev["q"], dev["k"], dev["v"], dev["do"], *out, causal, scale)
    return out


def _bnhd(t):
    """The same values stored as [B, N, H, d], viewed as [B, H, N, d]."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _compare(ref, got):
    (o0, l0, dq0, dk0, dv0), (o1, l1, dq1, dk1, dv1) = ref, got
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    assert gu.rel_l2(gu.to_f64(dq1), gu.to_f64(dq0)) < 1e-2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bnhd_layout_matches_contiguous(cuda_lib, d, causal):
    B, H, N = 2, 3, 300
    scale = gu.default_scale(d)
    dev, _ = gu.device_inputs(600 + d, B, H, N, d)
    ref = _contiguous_reference(cuda_lib, dev, causal, scale)
    q, k, v, do = (_bnhd(dev[n]) for n in ("q", "k", "v", "do"))
    o, dq, dk, dv = (_bnhd(torch.empty_like(dev["q"])) for _ in range(4))
    assert o.stride(2) == H * d  # really [B, N, H, d] in memory
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    _run(cuda_lib, q, k, v, do, o, lse, dq, dk, dv, causal, scale)
    _compare(ref, (o, lse, dq, dk, dv))


@pytest.mark.parametrize("causal", [False, True])
def test_packed_kv_matches_contiguous(cuda_lib, causal):
    """K and V interleaved per token in one [B, N, 2, H, d] buffer."""
    B, H, N, d = 2, 4, 520, 64
    scale = gu.default_scale(d)
    dev, _ = gu.device_inputs(650, B, H, N, d)
    ref = _contiguous_reference(cuda_lib, dev, causal, scale)
    kv = torch.stack([dev["k"].transpose(1, 2), dev["v"].transpose(1, 2)], dim=2).contiguous()
    k, v = kv[:, :, 0].transpose(1, 2), kv[:, :, 1].transpose(1, 2)
    assert k.stride(2) == 2 * H * d
    # the gradients of the packed buffer are written in the packed layout too
    dkv = torch.empty_like(kv)
    dk, dv = dkv[:, :, 0].transpose(1, 2), dkv[:, :, 1].transpose(1, 2)
    o, dq = torch.empty_like(dev["q"]), torch.empty_like(dev["q"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    _run(cuda_lib, dev["q"], k, v, dev["do"], o, lse, dq, dk, dv, causal, scale)
    _compare(ref, (o, lse, dq, dk, dv))


def test_bnhd_ragged_against_oracle(cuda_lib):
    B, H, N, d, causal = 1, 2, 233, 96, True
    scale = gu.default_scale(d)
    dev, bits = gu.device_inputs(660, B, H, N, d)
    q, k, v, do = (_bnhd(dev[n]) for n in ("q", "k", "v", "do"))
    o, dq, dk, dv = (_bnhd(torch.empty_like(dev["q"])) for _ in range(4))
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    _run(cuda_lib, q, k, v, do, o, lse, dq, dk, dv, causal, scale)
    for h in range(H):
        x = gu.head_f64(bits, 0, h)
        ow, lw = oracle.head_forward(x["q"], x["k"], x["v"], causal, scale)
        gu.check_o_lse(gu.to_f64(o[0, h]), gu.to_f64(lse[0, h]), ow, lw, f"head {h}")
        want = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
        gu.check_grads([gu.to_f64(g[0, h]) for g in (dq, dk, dv)], want, f"head {h}")

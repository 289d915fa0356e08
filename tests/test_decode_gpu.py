"""Decode parity: Nq <= 16 new rows per (batch, head) against a key/value cache
through fa_decode, against the fp64 oracle on each sequence's valid keys
(causal mask aligned at the bottom right). Covers one split and many splits
per head, per-sequence cache lengths (including 0 and fewer keys than
queries), a [B, Nk, H, d] cache layout and every head dimension.
"""

import numpy as np
import pytest

import oracle
from exact_tiled_attention_28_gb300 import inputs

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _decode(fa, seed, B, H, Nq, Nk, d, causal, seqlens=None, bnhd=False, scale=None):
    import torch
    scale = gu.default_scale(d) if scale is None else scale
    bits = inputs.nqnk_inputs(seed, B, H, Nq, Nk, d)
    dev = {n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()}
    x = {n: inputs.bf16_bits_to_f64(b) for n, b in bits.items()}
    k, v = dev["k"], dev["v"]
    if bnhd:  # the cache stored as [B, Nk, H, d]
        k = k.transpose(1, 2).contiguous().transpose(1, 2)
        v = v.transpose(1, 2).contiguous().transpose(1, 2)
    o = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    cs = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    ws = torch.full((fa.fa_decode_workspace_size(B, H, Nq, Nk, d),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    fa.fa_decode(dev["q"], k, v, o, lse, causal, scale, cache_seqlens=cs, workspace=ws)
    assert fa.fa_last_device_status() == fa.FA_OK
    og, lg = gu.to_f64(o), gu.to_f64(lse)
    what = f"B={B} H={H} Nq={Nq} Nk={Nk} d={d} causal={causal} seqlens={seqlens}"
    for b in range(B):
        nk = Nk if seqlens is None else seqlens[b]
        for h in range(H):
            ow, lw = oracle.head_forward(x["q"][b, h], x["k"][b, h, :nk], x["v"][b, h, :nk],
                                         causal, scale)
            empty = np.isneginf(lw)
            assert np.array_equal(np.isneginf(lg[b, h]), empty), what
            assert np.all(og[b, h][empty] == 0.0), what
            if np.any(~empty):
                gu.check_o_lse(og[b, h][~empty], lg[b, h][~empty], ow[~empty], lw[~empty],
                               f"{what} b={b} h={h}")
    return o, lse


@pytest.mark.parametrize("Nq", [1, 2, 3, 5, 8, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_many_splits(cuda_lib, Nq, causal):
    """Two heads: the keys of each are split over many CTAs."""
    _decode(cuda_lib, 500 + Nq, 1, 2, Nq, 5000, 128, causal)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_head_dims_and_cache_lengths(cuda_lib, d, causal):
    """Per-sequence cache lengths: 0 (no key), fewer keys than queries, a
    ragged tile, exactly one tile, the whole cache."""
    _decode(cuda_lib, 510 + d, 5, 3, 4, 1000, d, causal, seqlens=[0, 2, 129, 128, 1000])


@pytest.mark.parametrize("causal", [False, True])
def test_decode_one_split_per_head(cuda_lib, causal):
    """More heads than SMs: one CTA per head writes O and LSE directly."""
    _decode(cuda_lib, 520, 8, 24, 1, 700, 128, causal)
    _decode(cuda_lib, 521, 8, 24, 2, 300, 64, causal)


def test_decode_cache_layout_bnhd(cuda_lib):
    _decode(cuda_lib, 530, 3, 4, 2, 2000, 128, True, seqlens=[2000, 1, 777], bnhd=True)


def test_decode_matches_nqnk_path(cuda_lib):
    """The split decode and the tensor-core path for Nq != Nk compute the same
    function: their outputs agree to bf16 rounding."""
    import torch
    fa = cuda_lib
    B, H, Nq, Nk, d = 2, 4, 8, 3000, 128
    bits = inputs.nqnk_inputs(540, B, H, Nq, Nk, d)
    dev = {n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()}
    for causal in (False, True):
        o1 = torch.empty_like(dev["q"])
        l1 = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
        o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
        ws = torch.empty(fa.fa_decode_workspace_size(B, H, Nq, Nk, d), dtype=torch.uint8,
                         device="cuda")
        fa.fa_decode(dev["q"], dev["k"], dev["v"], o1, l1, causal, 0.1, workspace=ws)
        fa.fa_fwd(dev["q"], dev["k"], dev["v"], o2, l2, causal, 0.1)
        assert fa.fa_last_device_status() == fa.FA_OK
        assert gu.max_abs(gu.to_f64(l1), gu.to_f64(l2)) < 1e-4
        assert gu.rel_l2(gu.to_f64(o1), gu.to_f64(o2)) < 5e-3


def test_decode_cache_length_out_of_range_is_reported(cuda_lib):
    import torch
    fa = cuda_lib
    bits = inputs.nqnk_inputs(550, 2, 2, 1, 300, 64)
    dev = {n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()}
    o = torch.empty_like(dev["q"])
    lse = torch.empty((2, 2, 1), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fa_decode_workspace_size(2, 2, 1, 300, 64), dtype=torch.uint8,
                     device="cuda")
    cs = torch.tensor([300, 301], dtype=torch.int32, device="cuda")
    fa.fa_decode(dev["q"], dev["k"], dev["v"], o, lse, True, 0.1, cache_seqlens=cs, workspace=ws)
    assert fa.fa_last_device_status() == fa.FA_ERR_INVALID_ARG
    cs = torch.tensor([300, 299], dtype=torch.int32, device="cuda")
    fa.fa_decode(dev["q"], dev["k"], dev["v"], o, lse, True, 0.1, cache_seqlens=cs, workspace=ws)
    assert fa.fa_last_device_status() == fa.FA_OK


# More (batch, head) pairs than SMs and Nq >= 8: fa_decode runs the
# tensor-core forward over the dense batch with per-sequence key counts
# instead of the split-key kernel. B * H = 160 >= 152 SMs.

@pytest.mark.parametrize("Nq", [8, 13, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_tensor_core_path(cuda_lib, Nq, causal):
    rng = np.random.default_rng(560 + Nq)
    seqlens = [int(x) for x in rng.integers(1, 701, size=8)]
    seqlens[:3] = [0, Nq - 2, 700]  # no key, fewer keys than queries, the whole cache
    _decode(cuda_lib, 560 + Nq, 8, 20, Nq, 700, 128, causal, seqlens=seqlens)


@pytest.mark.parametrize("d", [32, 64, 96])
def test_decode_tensor_core_path_head_dims(cuda_lib, d):
    _decode(cuda_lib, 570 + d, 4, 40, 16, 300, d, True, seqlens=[300, 129, 5, 256])


def test_decode_tensor_core_path_uniform_cache_and_bnhd(cuda_lib):
    _decode(cuda_lib, 580, 8, 20, 9, 333, 128, True)
    _decode(cuda_lib, 581, 8, 20, 12, 1000, 64, False, seqlens=[1000, 1, 0, 999, 500, 128, 129, 2],
            bnhd=True)


def test_decode_tensor_core_path_bad_length_is_reported(cuda_lib):
    import torch
    fa = cuda_lib
    B, H, Nq, Nk, d = 8, 20, 8, 200, 64
    bits = inputs.nqnk_inputs(590, B, H, Nq, Nk, d)
    dev = {n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()}
    o = torch.empty_like(dev["q"])
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(fa.fa_decode_workspace_size(B, H, Nq, Nk, d), 16), dtype=torch.uint8,
                     device="cuda")
    cs = torch.tensor([200] * 7 + [-1], dtype=torch.int32, device="cuda")
    fa.fa_decode(dev["q"], dev["k"], dev["v"], o, lse, True, 0.1, cache_seqlens=cs, workspace=ws)
    assert fa.fa_last_device_status() == fa.FA_ERR_INVALID_ARG
    cs = torch.tensor([200] * 8, dtype=torch.int32, device="cuda")
    fa.fa_decode(dev["q"], dev["k"], dev["v"], o, lse, True, 0.1, cache_seqlens=cs, workspace=ws)
    assert fa.fa_last_device_status() == fa.FA_OK


@pytest.mark.parametrize("Nq", [1, 16])
def test_decode_bench_cache_sampled(cuda_lib, Nq):
    """The bench's decode cache (8192 keys, valid lengths in [4096, 8192],
    d = 128, H = 32) with B = 8, so that B * H still exceeds the SM count and
    both paths run in the bench's launch configuration: Nq = 1 the split-key
    kernel with one split per head, Nq = 16 the tensor-core forward. Every
    row finite; six sampled heads against the oracle."""
    import torch
    fa = cuda_lib
    B, H, Nk, d, causal = 8, 32, 8192, 128, True
    scale = gu.default_scale(d)
    seqlens = [int(n) for n in np.random.default_rng(9).integers(Nk // 2, Nk + 1, size=B)]
    bits = inputs.nqnk_inputs(595 + Nq, B, H, Nq, Nk, d)
    dev = {n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()}
    o = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    cs = torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(fa.fa_decode_workspace_size(B, H, Nq, Nk, d), 16), dtype=torch.uint8,
                     device="cuda")
    fa.fa_decode(dev["q"], dev["k"], dev["v"], o, lse, causal, scale, cache_seqlens=cs,
                 workspace=ws)
    assert fa.fa_last_device_status() == fa.FA_OK
    og, lg = gu.to_f64(o), gu.to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    for b, h in gu.sample_heads(B, H, 6, seed=Nq):
        nk = seqlens[b]
        x = {n: inputs.bf16_bits_to_f64(bits[n][b, h, :nk] if n != "q" else bits[n][b, h])
             for n in ("q", "k", "v")}
        ow, lw = oracle.head_forward(x["q"], x["k"], x["v"], causal, scale)
        gu.check_o_lse(og[b, h], lg[b, h], ow, lw, f"Nq={Nq} b={b} h={h} nk={nk}")


# Nq >= 8 with fewer (batch, head) pairs than SMs, at d = 64 and 128:
# fa_decode runs the tensor-core forward with the keys split by the decode
# plan (each split writes its normalised rows and log2 LSE), then merges the
# splits by log-sum-exp. Other head dimensions keep the split-key kernel.

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq", [8, 13, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_tensor_core_split_keys(cuda_lib, d, Nq, causal):
    """Per-sequence lengths: no key, fewer keys than queries, a ragged tile,
    the whole cache; splits past a short sequence's keys weigh nothing."""
    _decode(cuda_lib, 600 + d + Nq, 4, 3, Nq, 3000, d, causal, seqlens=[0, Nq - 3, 1025, 3000])


def test_decode_tensor_core_split_keys_uniform_and_bnhd(cuda_lib):
    _decode(cuda_lib, 610, 2, 5, 9, 4000, 128, True)
    _decode(cuda_lib, 611, 3, 4, 16, 2000, 64, False, seqlens=[2000, 1, 777], bnhd=True)


def test_decode_other_head_dims_keep_the_split_kernel(cuda_lib):
    _decode(cuda_lib, 612, 2, 3, 8, 1500, 96, True, seqlens=[1500, 300])
    _decode(cuda_lib, 613, 2, 3, 16, 1500, 32, False)


@pytest.mark.parametrize("Nq", [8, 16])
def test_decode_long_cache_few_heads_sampled(cuda_lib, Nq):
    """The bench's long-cache decode shape (B = 1, H = 32, a 131072-key cache
    with 93K valid keys, d = 128, causal) on the split tensor-core path: every
    row finite, four sampled heads against the oracle."""
    import torch
    fa = cuda_lib
    B, H, Nk, d, causal = 1, 32, 131072, 128, True
    scale = gu.default_scale(d)
    seqlens = [93162]
    bits = inputs.nqnk_inputs(620 + Nq, B, H, Nq, Nk, d)
    dev = {n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()}
    o = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    cs = torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    ws = torch.full((fa.fa_decode_workspace_size(B, H, Nq, Nk, d),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    fa.fa_decode(dev["q"], dev["k"], dev["v"], o, lse, causal, scale, cache_seqlens=cs,
                 workspace=ws)
    assert fa.fa_last_device_status() == fa.FA_OK
    og, lg = gu.to_f64(o), gu.to_f64(lse)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg))
    for b, h in gu.sample_heads(B, H, 4, seed=Nq):
        nk = seqlens[b]
        x = {n: inputs.bf16_bits_to_f64(bits[n][b, h, :nk] if n != "q" else bits[n][b, h])
             for n in ("q", "k", "v")}
        ow, lw = oracle.head_forward(x["q"], x["k"], x["v"], causal, scale)
        gu.check_o_lse(og[b, h], lg[b, h], ow, lw, f"Nq={Nq} b={b} h={h} nk={nk}")

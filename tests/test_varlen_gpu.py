"""Parity of sequences with unequal lengths through the C ABI against the fp64
oracle: dense batches with Nq != Nk (fa_fwd_nqnk / fa_bwd_nqnk) and packed
batches of variable-length sequences (fa_fwd_varlen / fa_bwd_varlen). Causal
masks are aligned at the bottom right; rows that see no key must come back
with O = 0 and LSE = -inf.
"""

import ctypes

import numpy as np
import pytest

import oracle
from exact_tiled_attention_28_gb300 import inputs

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _to_dev(bits):
    return {n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()}


def _f64(bits):
    return {n: inputs.bf16_bits_to_f64(b) for n, b in bits.items()}


def _check_fwd(o, lse, o_want, lse_want, what):
    """O/LSE parity; rows whose reference LSE is -inf must be O = 0, LSE = -inf."""
    empty = np.isneginf(lse_want)
    bad = np.argwhere(np.isneginf(lse) != empty)
    assert bad.size == 0, (f"{what}: rows without keys differ at {bad[:5].tolist()} "
                           f"(got {lse[tuple(bad[0])]}, want {lse_want[tuple(bad[0])]})")
    assert np.all(o[empty] == 0.0), f"{what}: O of a row without keys is not 0"
    if np.any(~empty):
        gu.check_o_lse(o[~empty], lse[~empty], o_want[~empty], lse_want[~empty], what)


# ---------------------------------------------------------------------------
# dense batches, Nq != Nk

def _nqnk(fa, seed, B, H, Nq, Nk, d, causal, scale=None):
    import torch
    scale = gu.default_scale(d) if scale is None else scale
    bits = inputs.nqnk_inputs(seed, B, H, Nq, Nk, d)
    dev, x = _to_dev(bits), _f64(bits)
    o = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd(dev["q"], dev["k"], dev["v"], o, lse, causal, scale)
    assert fa.fa_last_device_status() == fa.FA_OK
    ws = torch.full((fa.fa_bwd_workspace_size(B, H, Nq, d),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    dq = torch.full_like(dev["q"], float("nan"))
    dk = torch.full_like(dev["k"], float("nan"))
    dv = torch.full_like(dev["k"], float("nan"))
    fa.fa_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], dq, dk, dv, causal, scale, ws)
    assert fa.fa_last_device_status() == fa.FA_OK
    what = f"B={B} H={H} Nq={Nq} Nk={Nk} d={d} causal={causal}"
    o_want, lse_want = oracle.attention_forward(x["q"], x["k"], x["v"], causal, scale)
    _check_fwd(gu.to_f64(o), gu.to_f64(lse), o_want, lse_want, what)
    want = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
    gu.check_grads([gu.to_f64(t) for t in (dq, dk, dv)], want, what)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(200, 333), (333, 200), (1, 1000), (129, 1), (256, 640)])
def test_nqnk(cuda_lib, Nq, Nk, d, causal):
    _nqnk(cuda_lib, 300 + Nq + Nk, 2, 3, Nq, Nk, d, causal)


@pytest.mark.parametrize("d", [32, 96])
@pytest.mark.parametrize("causal", [False, True])
def test_nqnk_other_head_dims(cuda_lib, d, causal):
    _nqnk(cuda_lib, 310, 2, 2, 150, 300, d, causal)
    _nqnk(cuda_lib, 311, 1, 2, 300, 150, d, causal)


def test_nqnk_equal_lengths_match_dense_kernel_bitwise(cuda_lib):
    """Nq = Nk through fa_fwd_nqnk runs the same arithmetic in the same order
    as fa_fwd: the outputs agree bit for bit."""
    import torch
    fa = cuda_lib
    lib = fa.load()
    B, H, N, d = 2, 3, 300, 128
    for causal in (False, True):
        dev, _ = gu.device_inputs(320, B, H, N, d)
        o1, lse1 = gu.run_fwd(fa, dev, causal, 0.1)
        o2 = torch.full_like(o1, float("nan"))
        lse2 = torch.full_like(lse1, float("nan"))
        st = torch.cuda.current_stream().cuda_stream
        assert lib.fa_fwd_nqnk(dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(),
                               o2.data_ptr(), lse2.data_ptr(), B, H, N, N, d, None, int(causal),
                               0.1, st) == fa.FA_OK
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.equal(o1, o2) and torch.equal(lse1, lse2)


# ---------------------------------------------------------------------------
# packed batches

def _varlen(fa, seed, lens_q, lens_k, H, d, causal, scale=None, views=None, max_q=None,
            max_k=None):
    import torch
    scale = gu.default_scale(d) if scale is None else scale
    bits, cu_q, cu_k = inputs.packed_inputs(seed, lens_q, lens_k, H, d)
    x = _f64(bits)
    dev = _to_dev(bits) if views is None else views(_to_dev(bits))
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    mq = max(lens_q) if max_q is None else max_q
    mk = max(lens_k) if max_k is None else max_k
    o = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((H, Tq), float("nan"), dtype=torch.float32, device="cuda")
    fa.fa_fwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, cq, ck, mq, mk, causal, scale)
    assert fa.fa_last_device_status() == fa.FA_OK
    what = f"lens_q={lens_q} lens_k={lens_k} H={H} d={d} causal={causal}"
    o_want, lse_want = oracle.varlen_forward(x["q"], x["k"], x["v"], cu_q, cu_k, causal, scale)
    # the forward on its own, before the backward touches anything
    # (LSE is [H, T] while O is [T, H, d]: compare per (row, head))
    _check_fwd(gu.to_f64(o), gu.to_f64(lse).T, o_want, lse_want.T, "forward: " + what[-60:])
    ws = torch.full((fa.fa_bwd_varlen_workspace_size(len(lens_q), H, Tq, mk, d),), 0xFF,
                    dtype=torch.uint8, device="cuda")
    dq = torch.full_like(dev["q"], float("nan"))
    dk = torch.full_like(dev["k"], float("nan"))
    dv = torch.full_like(dev["k"], float("nan"))
    fa.fa_bwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], dq, dk, dv, cq, ck, mq, mk,
                     causal, scale, ws)
    assert fa.fa_last_device_status() == fa.FA_OK
    # the backward leaves the forward's outputs alone
    _check_fwd(gu.to_f64(o), gu.to_f64(lse).T, o_want, lse_want.T, "after backward: " + what[-60:])
    want = oracle.varlen_backward(x["q"], x["k"], x["v"], x["do"], cu_q, cu_k, causal, scale)
    gu.check_grads([gu.to_f64(t) for t in (dq, dk, dv)], want, what)
    return o, lse


# empty sequences on either side, Nq > Nk (rows without keys), Nq = 1, equal lengths
LENS_Q = [130, 0, 257, 1, 64, 300, 128]
LENS_K = [200, 5, 257, 129, 0, 100, 128]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen(cuda_lib, d, causal):
    _varlen(cuda_lib, 400, LENS_Q, LENS_K, 2, d, causal)


@pytest.mark.parametrize("d", [32, 96])
def test_varlen_other_head_dims(cuda_lib, d):
    _varlen(cuda_lib, 401, LENS_Q, LENS_K, 2, d, True)


def test_varlen_strided_views(cuda_lib):
    """Rows of q, o, dO, dq wider than H * d (a buffer with a spare head) and
    K, V as halves of one [T, 2, H, d] buffer go through the strided form."""
    import torch

    def views(dev):
        out = {}
        for n in ("q", "do"):
            t = dev[n]
            buf = torch.zeros(t.shape[0], t.shape[1] + 1, t.shape[2], dtype=t.dtype, device="cuda")
            buf[:, 1:] = t
            out[n] = buf[:, 1:]
        kv = torch.stack([dev["k"], dev["v"]], dim=1)
        out["k"], out["v"] = kv[:, 0], kv[:, 1]
        return out

    for causal in (False, True):
        _varlen(cuda_lib, 402, [100, 300, 7], [250, 300, 1], 3, 128, causal, views=views)


def test_varlen_long_batch(cuda_lib):
    """Eight sequences of up to 2048 tokens, four heads: many CTAs of the
    persistent grid on sequences of different lengths."""
    rng = np.random.default_rng(403)
    lens = [int(x) for x in rng.integers(1, 2049, size=8)]
    for causal in (False, True):
        _varlen(cuda_lib, 403, lens, lens, 4, 128, causal)


def test_varlen_uniform_matches_dense_kernel_bitwise(cuda_lib):
    """A packed batch of equal-length sequences runs the same arithmetic as the
    dense kernel on the same values: O and LSE agree bit for bit."""
    import torch
    fa = cuda_lib
    B, H, N, d = 3, 2, 300, 64
    for causal in (False, True):
        dev, _ = gu.device_inputs(404, B, H, N, d)
        o1, lse1 = gu.run_fwd(fa, dev, causal, 0.125)
        pq, pk, pv = (dev[n].transpose(1, 2).reshape(B * N, H, d).contiguous()
                      for n in ("q", "k", "v"))
        cu = torch.arange(0, B * N + 1, N, dtype=torch.int32, device="cuda")
        o2 = torch.empty_like(pq)
        lse2 = torch.empty((H, B * N), dtype=torch.float32, device="cuda")
        fa.fa_fwd_varlen(pq, pk, pv, o2, lse2, cu, cu, N, N, causal, 0.125)
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.equal(o2.reshape(B, N, H, d).transpose(1, 2), o1)
        assert torch.equal(lse2.reshape(H, B, N).transpose(0, 1), lse1)


def test_varlen_malformed_offsets_are_reported(cuda_lib):
    """Offsets whose last entry is not total_q, or a length above
    max_seqlen_q, are reported as FA_ERR_INVALID_ARG by the next status read;
    the offsets stay inside [0, total], and the kernels clamp every access."""
    import torch
    fa = cuda_lib
    H, d = 2, 64
    bits, cu_q, cu_k = inputs.packed_inputs(405, [100, 200], [150, 150], H, d)
    dev = _to_dev(bits)
    o = torch.empty_like(dev["q"])
    lse = torch.empty((H, 300), dtype=torch.float32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    short = torch.tensor([0, 100, 250], dtype=torch.int32, device="cuda")
    fa.fa_fwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, short, ck, 200, 150, True, 0.1)
    assert fa.fa_last_device_status() == fa.FA_ERR_INVALID_ARG
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    fa.fa_fwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, cq, ck, 150, 150, True, 0.1)
    assert fa.fa_last_device_status() == fa.FA_ERR_INVALID_ARG
    fa.fa_fwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, cq, ck, 200, 150, True, 0.1)
    assert fa.fa_last_device_status() == fa.FA_OK


@pytest.mark.parametrize("n_seq,d", [(700, 64), (5000, 64), (5000, 128)])
def test_varlen_many_short_sequences(cuda_lib, n_seq, d):
    """Many short sequences, some empty, most in one level class of the
    compacted schedule, which every CTA of the forward builds for itself (at
    d = 64 both sizes fit in its shared memory; at d = 128 the 5000 do not and
    the forward takes the uncompacted order; the backward always builds its
    schedule once, in the workspace). A second forward gives the same bits."""
    import torch
    rng = np.random.default_rng(406 + n_seq)
    lens_q = [int(x) for x in rng.integers(0, 40, size=n_seq)]
    lens_k = [int(x) for x in rng.integers(0, 40, size=n_seq)]
    lens_k[0] = max(lens_k[0], 1)
    for causal in (False, True):
        o, lse = _varlen(cuda_lib, 406, lens_q, lens_k, 1, d, causal)
        bits, cu_q, cu_k = inputs.packed_inputs(406, lens_q, lens_k, 1, d)
        dev = _to_dev(bits)
        cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
        ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
        o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
        cuda_lib.fa_fwd_varlen(dev["q"], dev["k"], dev["v"], o2, lse2, cq, ck, max(lens_q),
                               max(lens_k), causal, gu.default_scale(d))
        assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_bench_batch_sampled(cuda_lib, causal):
    """The bench's packed batch (16 sequences of 276..3885 tokens, H = 16,
    d = 128): every output finite, and three sampled (sequence, head) blocks
    against the oracle, forward and backward (sequences are independent)."""
    import torch
    fa = cuda_lib
    lens = [int(n) for n in np.random.default_rng(7).integers(256, 4097, size=16)]
    H, d = 16, 128
    scale = gu.default_scale(d)
    bits, cu_q, cu_k = inputs.packed_inputs(420, lens, lens, H, d)
    dev = _to_dev(bits)
    T = int(cu_q[-1])
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    o = torch.empty_like(dev["q"])
    lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
    fa.fa_fwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, cq, cq, max(lens), max(lens), causal,
                     scale)
    ws = torch.empty(fa.fa_bwd_varlen_workspace_size(16, H, T, max(lens), d), dtype=torch.uint8,
                     device="cuda")
    dq, dk, dv = (torch.empty_like(dev["q"]) for _ in range(3))
    fa.fa_bwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], dq, dk, dv, cq, cq,
                     max(lens), max(lens), causal, scale, ws)
    assert fa.fa_last_device_status() == fa.FA_OK
    g = {n: gu.to_f64(t) for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    for t in g.values():
        assert np.all(np.isfinite(t))
    rng = np.random.default_rng(421)
    for b, h in [(int(rng.integers(16)), int(rng.integers(H))) for _ in range(3)]:
        r0, r1 = int(cu_q[b]), int(cu_q[b + 1])
        x = {n: inputs.bf16_bits_to_f64(bits[n][r0:r1, h]) for n in ("q", "k", "v", "do")}
        ow, lw = oracle.head_forward(x["q"], x["k"], x["v"], causal, scale)
        gu.check_o_lse(g["o"][r0:r1, h], g["lse"][h, r0:r1], ow, lw, f"b={b} h={h}")
        want = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
        gu.check_grads((g["dq"][r0:r1, h], g["dk"][r0:r1, h], g["dv"][r0:r1, h]), want,
                       f"b={b} h={h} n={r1 - r0}")

"""fa_bwd_noalloc, the backward for callers that cannot allocate device memory
(their memory is all in their own pool, or they must not call cudaMalloc
while running). Through the C ABI, on two calls in a row sharing its fixed
scratch array, it must give what fa_bwd gives and match the fp64 oracle. The
head dimensions 64 and 128 run the d <= 128 kernels; d = 256 runs its own
dK/dV kernel over the same workspace layout, and N = 200 leaves ragged tiles
and padded D / lse rows. This file is collected last so that a stop at its
first failure has already run every other test."""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_28_gb300 import binding

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _ptrs(ts):
    return [t.data_ptr() for t in ts]


def _noalloc(fa, dev, o, lse, B, H, N, d, causal, scale):
    stream = torch.cuda.current_stream().cuda_stream
    grads = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]
    st = binding.fa_bwd_noalloc_raw(*_ptrs([dev["q"], dev["k"], dev["v"], o, lse, dev["do"]]),
                                    *_ptrs(grads), B, H, N, d, causal, scale, stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert fa.fa_last_device_status() == fa.FA_OK
    return [gu.to_f64(g) for g in grads]


def _check_twice(fa, seed, B, H, N, d, causal, heads=None):
    """Two no-alloc calls against fa_bwd (dK, dV bit for bit: no atomics) and
    against the oracle on the given (b, h) heads (all when None)."""
    scale = gu.default_scale(d)
    dev, bits = gu.device_inputs(seed, B, H, N, d)
    o, lse = gu.run_fwd(fa, dev, causal, scale)
    want = [gu.to_f64(g) for g in gu.run_bwd(fa, dev, o, lse, causal, scale)]
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    ref = {}
    for b, h in heads:
        x = gu.head_f64(bits, b, h)
        ref[(b, h)] = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
    for call in range(2):
        got = _noalloc(fa, dev, o, lse, B, H, N, d, causal, scale)
        for name, g, w in zip(("dQ", "dK", "dV"), got, want):
            assert np.all(np.isfinite(g)), f"call {call}: non-finite {name}"
            rl = gu.rel_l2(g, w)
            assert rl <= gu.TOL_GRAD_RELL2, f"call {call}: {name} vs fa_bwd rel-L2 {rl:.3e}"
        assert np.array_equal(got[1], want[1]) and np.array_equal(got[2], want[2])
        for (b, h), r in ref.items():
            gu.check_grads([g[b, h] for g in got], r,
                           f"call {call}, head ({b},{h}) vs the oracle, N={N} d={d}")


@pytest.mark.parametrize("B,H,N,d,causal", [(4, 8, 1024, 64, True), (2, 3, 383, 128, False),
                                            (1, 2, 200, 256, True), (1, 2, 200, 256, False)])
def test_noalloc_matches_fa_bwd_and_oracle_twice(cuda_lib, B, H, N, d, causal):
    heads = None if B * H <= 8 else gu.sample_heads(B, H, 3, seed=N)
    _check_twice(cuda_lib, 500 + N + d, B, H, N, d, causal, heads)


def test_noalloc_near_its_limit_after_a_smaller_call(cuda_lib):
    """A call whose workspace fills 95% of the array, right after a small
    one: every byte the large call reads was rewritten by it, not left over."""
    fa = cuda_lib
    B, H, N, d = 1, 15, 4096, 128
    need = fa.fa_bwd_workspace_size(B, H, N, d)
    assert 0.9 * binding.NOALLOC_SCRATCH_BYTES < need <= binding.NOALLOC_SCRATCH_BYTES
    assert fa.fa_bwd_workspace_size(B, H + 1, N, d) > binding.NOALLOC_SCRATCH_BYTES
    _check_twice(fa, 900, 1, 2, 300, 64, True)
    _check_twice(fa, 901, B, H, N, d, False, heads=[(0, 0), (0, H - 1)])


def test_noalloc_refuses_sizes_beyond_its_scratch(cuda_lib):
    fa = cuda_lib
    B, H, N, d = 1, 16, 32768, 128
    assert fa.fa_bwd_workspace_size(B, H, N, d) > binding.NOALLOC_SCRATCH_BYTES
    fake = 4096  # never dereferenced: the size check comes first
    st = binding.fa_bwd_noalloc_raw(*([fake] * 9), B, H, N, d, True, 0.1, None)
    assert st == fa.FA_ERR_WORKSPACE
    st = binding.fa_bwd_noalloc_raw(*([fake] * 9), 1, 16, 4096, 128, False, 0.1, None)
    assert st == fa.FA_ERR_WORKSPACE

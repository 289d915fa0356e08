"""fa_bwd_noalloc, the backward for callers that cannot allocate device memory
(their memory is all in their own pool, or they must not call cudaMalloc
while running). It must give what fa_bwd gives, through the C ABI, on two
calls in a row sharing its fixed scratch array. This file is collected last
so that a stop at its first failure has already run every other test."""

import numpy as np
import pytest
import torch

from exact_tiled_attention_28_gb300 import binding

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _ptrs(ts):
    return [t.data_ptr() for t in ts]


@pytest.mark.parametrize("B,H,N,d,causal", [(4, 8, 1024, 64, True), (2, 3, 383, 128, False)])
def test_noalloc_matches_fa_bwd_twice(cuda_lib, B, H, N, d, causal):
    fa = cuda_lib
    scale = gu.default_scale(d)
    dev, _ = gu.device_inputs(500 + N, B, H, N, d)
    o, lse = gu.run_fwd(fa, dev, causal, scale)
    want = [gu.to_f64(g) for g in gu.run_bwd(fa, dev, o, lse, causal, scale)]
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        grads = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]
        st = binding.fa_bwd_noalloc_raw(*_ptrs([dev["q"], dev["k"], dev["v"], o, lse, dev["do"]]),
                                        *_ptrs(grads), B, H, N, d, causal, scale, stream)
        assert st == fa.FA_OK, fa.fa_status_string(st)
        assert fa.fa_last_device_status() == fa.FA_OK
        got = [gu.to_f64(g) for g in grads]
        for name, g, w in zip(("dQ", "dK", "dV"), got, want):
            assert np.all(np.isfinite(g)), f"call {call}: non-finite {name}"
            rl = gu.rel_l2(g, w)
            assert rl <= gu.TOL_GRAD_RELL2, f"call {call}: {name} rel-L2 {rl:.3e}"
        # dK and dV involve no atomics: the same kernel gives the same bits
        assert np.array_equal(got[1], want[1]) and np.array_equal(got[2], want[2])


def test_noalloc_refuses_sizes_beyond_its_scratch(cuda_lib):
    fa = cuda_lib
    B, H, N, d = 1, 16, 32768, 128
    assert fa.fa_bwd_workspace_size(B, H, N, d) > binding.NOALLOC_SCRATCH_BYTES
    fake = 4096  # never dereferenced: the size check comes first
    st = binding.fa_bwd_noalloc_raw(*([fake] * 9), B, H, N, d, True, 0.1, None)
    assert st == fa.FA_ERR_WORKSPACE

"""The debug build (libfa_debug.so: the same sources with FA_DEBUG) on the GPU.

1. Index checks. Its kernels check the index range of their global stores; on
   valid inputs no check may fire, and the parity results are those of the
   release build. A self-test kernel whose one check fails shows that a
   failed check reaches fa_last_device_status as FA_ERR_DEVICE_CHECK.
2. The abort path of the real attention kernels, made to run without a GPU
   fault: with the bounded-wait limit set to 0 (fa_set_wait_limit_ns), every
   on-chip wait that does not complete at its first try gives up, so each
   kernel's roles stop, wait (bounded) for their copies in flight, release
   tensor memory and exit, and the kernel records FA_ERR_TIMEOUT. The test
   then restores the 2 s limit and runs the same call again on the same
   context: its results must match the fp64 oracle, which also shows that the
   aborted kernels freed their tensor memory (an allocation that never
   returns would time out).

Covered by the abort tests: the forward at d = 64 (causal, dense
instantiation) and d = 128 (non-causal, equal-length instantiation), the
backward's dK/dV kernel at d = 64 and 128 with either dQ path (so also the
separate dQ kernel), the d = 256 forward and dK/dV kernels, and the packed
variable-length forward and backward.

A wait gives up only if its first try does not complete, and a first try
suspends the thread for a hardware-dependent time before it returns. The
items here are long (16 key tiles and more), so that waits spanning a whole
item (the loader's wait for the next item's buffers, the epilogue's wait for
the last product) outlast that time. The split-key decode kernel is not
covered: each of its waits spans one 128-key tile (about 1 to 2 us), and on
GB300 every first try completed, so no wait of it gave up at limit 0.

The file is collected after the parity tests (and before the no-alloc test,
which comes last), so a run that stops at a first failure has checked parity
before it makes any kernel give up.
"""

import pytest

import oracle
from exact_tiled_attention_28_gb300 import binding, inputs

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture
def dbg(cuda_lib):
    """The binding routed through libfa_debug.so for one test."""
    before = cuda_lib.use_library(True)
    assert cuda_lib.fa_is_debug_build()
    assert cuda_lib.fa_last_device_status() == cuda_lib.FA_OK
    try:
        yield cuda_lib
    finally:
        cuda_lib.use_library(before)


def test_failed_index_check_is_reported(dbg):
    dbg.fa_selftest_index_check()
    assert dbg.fa_last_device_status() == dbg.FA_ERR_DEVICE_CHECK
    assert dbg.fa_last_device_status() == dbg.FA_OK


@pytest.mark.parametrize("d,causal", [(64, True), (128, False), (96, True), (256, False)])
def test_debug_build_parity_and_no_check_fires(dbg, d, causal):
    """Ragged N (a partial last tile), several heads: forward and backward
    through the debug kernels match the oracle, and no index check fires."""
    from .test_bwd_gpu import _full_check as bwd_check
    from .test_fwd_gpu import _full_check as fwd_check
    fwd_check(dbg, 800 + d, 2, 3, 333, d, causal)
    bwd_check(dbg, 810 + d, 2, 3, 333, d, causal)
    assert dbg.fa_last_device_status() == dbg.FA_OK


@pytest.mark.parametrize("causal", [False, True])
def test_debug_build_other_paths_no_check_fires(dbg, causal):
    """The separate dQ kernel, strided [B, N, H, d] tensors, a packed batch and
    decode through the debug kernels: results as the release build's tests
    require, and no index check fires."""
    import torch
    from .test_dq_path_gpu import _check as dq_check
    from .test_decode_gpu import _decode
    from .test_layouts_gpu import test_bnhd_ragged_against_oracle, test_packed_kv_matches_contiguous
    from .test_varlen_gpu import _varlen
    dq_check(dbg, 820, 1, 3, 700, 128, causal)
    test_bnhd_ragged_against_oracle(dbg)
    test_packed_kv_matches_contiguous(dbg, causal)
    _varlen(dbg, 830, [130, 0, 257, 1], [200, 5, 257, 129], 2, 64, causal)
    _decode(dbg, 840, 3, 2, 2, 1500, 128, causal, seqlens=[0, 77, 1500])
    assert dbg.fa_last_device_status() == dbg.FA_OK
    torch.cuda.synchronize()


def _abort_then_recover(fa, run, check):
    """run() enqueues one call; returns after checking the timeout record of
    the aborted run and the results of a normal run."""
    assert fa.fa_last_device_status() == fa.FA_OK
    fa.fa_set_wait_limit_ns(0)
    try:
        run()
        st = fa.fa_last_device_status()
    finally:
        fa.fa_set_wait_limit_ns(binding.WAIT_LIMIT_NS_DEFAULT)
    assert st == fa.FA_ERR_TIMEOUT, (
        f"status {fa.fa_status_string(st)}: no wait gave up with the limit at 0")
    assert fa.fa_last_device_status() == fa.FA_OK  # reading cleared the record
    run()
    assert fa.fa_last_device_status() == fa.FA_OK
    check()


def _dense_inputs(seed, B, H, N, d):
    import torch
    dev, bits = gu.device_inputs(seed, B, H, N, d)
    o = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    return dev, bits, o, lse


@pytest.mark.parametrize("d,causal", [(64, True), (128, False), (256, False)])
def test_forward_aborts_and_recovers(dbg, d, causal):
    fa = dbg
    B, H, N = 1, 3, 2048
    scale = gu.default_scale(d)
    dev, bits, o, lse = _dense_inputs(40 + d, B, H, N, d)

    def run():
        fa.fa_fwd(dev["q"], dev["k"], dev["v"], o, lse, causal, scale)

    def check():
        for b, h in ((0, 0), (B - 1, H - 1)):
            x = gu.head_f64(bits, b, h)
            ow, lw = oracle.head_forward(x["q"], x["k"], x["v"], causal, scale)
            gu.check_o_lse(gu.to_f64(o[b, h]), gu.to_f64(lse[b, h]), ow, lw,
                           f"forward d={d} head ({b},{h}) after an aborted call")

    _abort_then_recover(fa, run, check)


@pytest.mark.parametrize("d,causal,dq_path", [(64, True, 1), (128, False, 1), (128, True, 1),
                                               (256, True, 1), (128, False, 2), (64, True, 2)])
def test_backward_aborts_and_recovers(dbg, d, causal, dq_path):
    """dq_path 1: the dK/dV kernel with atomic dQ; 2: the dK/dV kernel without
    dQ and the separate, query-stationary dQ kernel."""
    import torch
    fa = dbg
    B, H, N = 1, 3, 2048
    scale = gu.default_scale(d)
    dev, bits, _, _ = _dense_inputs(60 + d, B, H, N, d)
    o, lse = gu.run_fwd(fa, dev, causal, scale)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    grads = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]

    def run():
        fa.fa_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], *grads, causal, scale, ws,
                  dq_path=dq_path)

    def check():
        for h in (0, H - 1):
            x = gu.head_f64(bits, 0, h)
            want = oracle.head_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
            gu.check_grads([gu.to_f64(g[0, h]) for g in grads], want,
                           f"backward d={d} head {h} after an aborted call")

    _abort_then_recover(fa, run, check)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_batch_aborts_and_recovers(dbg, causal):
    import torch
    fa = dbg
    H, d = 2, 128
    lens = [300, 1, 2100, 130]
    scale = gu.default_scale(d)
    bits, cu_q, _ = inputs.packed_inputs(70, lens, lens, H, d)
    dev = {n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()}
    x = {n: inputs.bf16_bits_to_f64(b) for n, b in bits.items()}
    cu = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    T, mx = int(cu_q[-1]), max(lens)
    o = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    grads = [torch.full_like(dev["q"], float("nan")) for _ in range(3)]
    ws = torch.empty(fa.fa_bwd_varlen_workspace_size(len(lens), H, T, mx, d), dtype=torch.uint8,
                     device="cuda")

    def run():
        fa.fa_fwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, cu, cu, mx, mx, causal, scale)
        fa.fa_bwd_varlen(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], *grads, cu, cu, mx, mx,
                         causal, scale, ws)

    def check():
        ow, lw = oracle.varlen_forward(x["q"], x["k"], x["v"], cu_q, cu_q, causal, scale)
        gu.check_o_lse(gu.to_f64(o), gu.to_f64(lse), ow, lw, "packed forward after an abort")
        want = oracle.varlen_backward(x["q"], x["k"], x["v"], x["do"], cu_q, cu_q, causal, scale)
        gu.check_grads([gu.to_f64(g) for g in grads], want, "packed backward after an abort")

    _abort_then_recover(fa, run, check)


def test_wait_limit_rejects_values_above_the_default(dbg):
    with pytest.raises(dbg.FaError):
        dbg.fa_set_wait_limit_ns(binding.WAIT_LIMIT_NS_DEFAULT + 1)
    dbg.fa_set_wait_limit_ns(binding.WAIT_LIMIT_NS_DEFAULT)


def test_release_build_has_no_debug_hooks(cuda_lib):
    assert not cuda_lib.fa_is_debug_build()
    with pytest.raises(cuda_lib.FaError) as e:
        cuda_lib.fa_set_wait_limit_ns(0)
    assert e.value.status == cuda_lib.FA_ERR_UNSUPPORTED

"""The entry points under CUDA graph capture. Every call only enqueues work
on its stream: tensor maps travel as kernel parameters, the workspaces are
the caller's, and nothing synchronises. So a caller can capture fa_fwd,
fa_bwd, the packed-batch pair and fa_decode into a CUDA graph once and
replay it, without the per-call host work. Replays must write what eager
calls write (bit for bit, except dq, whose fp32 atomic sums may round
differently in their last bf16 bit), and must read the buffers as they are
at replay time: new values copied into the same inputs give the eager
result for those values."""

import pytest
import torch

from exact_tiled_attention_28_gb300 import inputs

from . import gpu_util as gu

pytestmark = pytest.mark.gpu


def _capture(fn):
    """fn() captured into a CUDA graph (after one run on a side stream, the
    pattern capture expects for first-use work)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _snapshot(outs):
    return {n: t.clone() for n, t in outs.items()}


def _poison(outs):
    for t in outs.values():
        if t.dtype == torch.uint8:
            continue
        t.fill_(float("nan"))


def _same(got, want, what, atomic=("dq",)):
    for n, t in want.items():
        g = got[n]
        if n in atomic:
            # fp32 atomic sums: the order of additions may differ per run
            num = torch.linalg.vector_norm((g.float() - t.float()).flatten())
            den = torch.linalg.vector_norm(t.float().flatten())
            assert torch.isfinite(g.float()).all(), f"{what}: {n} has non-finite values"
            assert (num / den).item() <= 1e-3, f"{what}: {n} rel-L2 {num / den:.2e}"
        else:
            assert torch.equal(g, t), f"{what}: {n} differs from the eager call"


def _replay_matches_eager(fa, run, outs, set_inputs, what):
    """run() eagerly, capture it, replay twice over poisoned outputs, then
    replay on new input values and compare with an eager run on those."""
    set_inputs(0)
    run()
    assert fa.fa_last_device_status() == fa.FA_OK
    want = _snapshot(outs)
    g = _capture(run)
    for rep in range(2):
        _poison(outs)
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
        _same(outs, want, f"{what}, replay {rep}")
    set_inputs(1)
    _poison(outs)
    g.replay()
    torch.cuda.synchronize()
    replayed = _snapshot(outs)
    _poison(outs)
    run()
    assert fa.fa_last_device_status() == fa.FA_OK
    _same(replayed, _snapshot(outs), f"{what}, new inputs")
    assert not torch.equal(replayed["o"], want["o"]), f"{what}: replay ignored new inputs"
    del g


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 2, 300, 128, False), (2, 3, 384, 64, True),
                                            (1, 2, 200, 256, True), (1, 2, 130, 32, False)])
def test_dense_fwd_bwd_graph(cuda_lib, B, H, N, d, causal):
    fa = cuda_lib
    scale = gu.default_scale(d)
    srcs = [{n: inputs.bits_to_torch_bf16(b).cuda()
             for n, b in inputs.attention_inputs(seed, B, H, N, d).items()} for seed in (31, 32)]
    x = {n: torch.empty_like(t) for n, t in srcs[0].items()}
    outs = {"o": torch.empty_like(x["q"]),
            "lse": torch.empty((B, H, N), dtype=torch.float32, device="cuda"),
            "dq": torch.empty_like(x["q"]), "dk": torch.empty_like(x["q"]),
            "dv": torch.empty_like(x["q"])}
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")

    def set_inputs(i):
        for n in x:
            x[n].copy_(srcs[i][n])

    def run():
        fa.fa_fwd(x["q"], x["k"], x["v"], outs["o"], outs["lse"], causal, scale)
        fa.fa_bwd(x["q"], x["k"], x["v"], outs["o"], outs["lse"], x["do"], outs["dq"],
                  outs["dk"], outs["dv"], causal, scale, ws)

    _replay_matches_eager(fa, run, outs, set_inputs,
                          f"B={B} H={H} N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_fwd_bwd_graph(cuda_lib, causal):
    fa = cuda_lib
    lens, H, d = [100, 257, 31, 140], 2, 64
    scale = gu.default_scale(d)
    srcs = []
    for seed in (41, 42):
        bits, cu, _ = inputs.packed_inputs(seed, lens, lens, H, d)
        srcs.append({n: inputs.bits_to_torch_bf16(b).cuda() for n, b in bits.items()})
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    T, mx = int(cu[-1]), max(lens)
    x = {n: torch.empty_like(t) for n, t in srcs[0].items()}
    outs = {"o": torch.empty_like(x["q"]),
            "lse": torch.empty((H, T), dtype=torch.float32, device="cuda"),
            "dq": torch.empty_like(x["q"]), "dk": torch.empty_like(x["k"]),
            "dv": torch.empty_like(x["k"])}
    ws = torch.empty(fa.fa_bwd_varlen_workspace_size(len(lens), H, T, mx, d), dtype=torch.uint8,
                     device="cuda")

    def set_inputs(i):
        for n in x:
            x[n].copy_(srcs[i][n])

    def run():
        fa.fa_fwd_varlen(x["q"], x["k"], x["v"], outs["o"], outs["lse"], cu_t, cu_t, mx, mx,
                         causal, scale)
        fa.fa_bwd_varlen(x["q"], x["k"], x["v"], outs["o"], outs["lse"], x["do"], outs["dq"],
                         outs["dk"], outs["dv"], cu_t, cu_t, mx, mx, causal, scale, ws)

    _replay_matches_eager(fa, run, outs, set_inputs, f"packed lens={lens} causal={causal}")


@pytest.mark.parametrize("Nq", [1, 8])
def test_decode_graph(cuda_lib, Nq):
    fa = cuda_lib
    B, H, Nk, d = 3, 2, 700, 128
    scale = gu.default_scale(d)
    srcs = [{n: inputs.bits_to_torch_bf16(b).cuda()
             for n, b in inputs.nqnk_inputs(seed, B, H, Nq, Nk, d).items()} for seed in (51, 52)]
    x = {n: torch.empty_like(t) for n, t in srcs[0].items()}
    cs = torch.tensor([700, 333, 1], dtype=torch.int32, device="cuda")
    outs = {"o": torch.empty_like(x["q"]),
            "lse": torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")}
    ws = torch.empty(fa.fa_decode_workspace_size(B, H, Nq, Nk, d), dtype=torch.uint8,
                     device="cuda")

    def set_inputs(i):
        for n in x:
            x[n].copy_(srcs[i][n])

    def run():
        fa.fa_decode(x["q"], x["k"], x["v"], outs["o"], outs["lse"], True, scale,
                     cache_seqlens=cs, workspace=ws)

    _replay_matches_eager(fa, run, outs, set_inputs, f"decode Nq={Nq}")

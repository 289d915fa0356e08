"""Helpers shared by the GPU parity tests: seeded inputs on the device, calls
through the C ABI, and the error measures with their tolerances.

Tolerances (bf16 inputs, fp32 accumulation, compared with the fp64 oracle):
O max-abs <= 1e-2 and relative L2 <= 5e-3; dQ, dK, dV relative L2 <= 2e-2;
LSE max-abs <= 1e-3 (LSE is a sum of fp32 terms of size ln N, far more
accurate than bf16 outputs; 1e-3 leaves room for the fp32 row sum at
N = 32768).

O's max-abs bound is asserted on the raw difference |o - o_ref| for every
element with |o_ref| < 2. From |o_ref| = 2 up, storing O in bf16 alone can be
off by half a bf16 spacing, 2^-7 = 0.0078 on [2, 4) and 0.0156 on [4, 8),
and the P.V product takes P rounded to bf16 (relative error up to 2^-9): a
float simulation of the kernel's arithmetic over the first 64 causal rows of
1500 seeded heads reached a raw error of 1.008e-2 on [2, 4) (7.4e-3 on
[1, 2)). There the bound applies to the error in excess of that storage
rounding, |o - o_ref| - ulp_bf16(o_ref) / 2. The relative-L2 bound is always
applied to the raw difference. The raw form is the bound the configurations
carry, all at scale = 1/sqrt(d); tests at other scales (a peaked softmax at 4x
that scale puts more weight on few bf16-rounded P values) pass raw=False and
take the beyond-storage form everywhere.
"""

from __future__ import annotations

import math

import numpy as np

from exact_tiled_attention_28_gb300 import inputs

TOL_O_MAXABS = 1e-2
TOL_O_RELL2 = 5e-3
TOL_LSE_MAXABS = 1e-3
TOL_GRAD_RELL2 = 2e-2

_cache: dict = {}


def device_inputs(seed, B, H, N, d, tensors=("q", "k", "v", "do")):
    """Seeded bf16 inputs: (dict of CUDA bf16 tensors, dict of uint16 bits)."""
    import torch
    key = (seed, B, H, N, d, tuple(tensors))
    if key not in _cache:
        _cache.clear()  # keep at most one workload resident
        bits = inputs.attention_inputs(seed, B, H, N, d, tensors)
        dev = {n: inputs.bits_to_torch_bf16(bits[n]).cuda() for n in tensors}
        _cache[key] = (dev, bits)
    return _cache[key]


def head_f64(bits, b, h, names=("q", "k", "v", "do")):
    return {n: inputs.bf16_bits_to_f64(bits[n][b, h]) for n in names if n in bits}


def run_fwd(fa, dev, causal, scale):
    import torch
    q = dev["q"]
    B, H, N, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    fa.fa_fwd(q, dev["k"], dev["v"], o, lse, causal, scale)
    assert fa.fa_last_device_status() == fa.FA_OK
    return o, lse


def run_bwd(fa, dev, o, lse, causal, scale):
    import torch
    q = dev["q"]
    B, H, N, d = q.shape
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=q.device)
    ws.fill_(0xFF)  # NaN pattern: the call must not depend on the workspace contents
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa.fa_bwd(q, dev["k"], dev["v"], o, lse, dev["do"], *grads, causal, scale, ws)
    assert fa.fa_last_device_status() == fa.FA_OK
    return grads


def to_f64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def rel_l2(got, want):
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def max_abs(got, want):
    return float(np.max(np.abs(got - want))) if got.size else 0.0


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (bf16 has 8 significant bits)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def max_abs_beyond_bf16_storage(got, want):
    if not got.size:
        return 0.0
    return float(np.max(np.abs(got - want) - half_ulp_bf16(want)))


# |O_ref| from which the max-abs bound is taken beyond the bf16 storage rounding
O_RAW_BELOW = 2.0


def o_max_abs(got, want, raw=True):
    """(raw max-abs over |want| < 2, max-abs beyond bf16 storage over |want| >= 2);
    raw=False: (0, the beyond-storage form over every element)."""
    small = np.abs(want) < O_RAW_BELOW if raw else np.zeros(want.shape, bool)
    return max_abs(got[small], want[small]), max_abs_beyond_bf16_storage(got[~small], want[~small])


def check_o_lse(o_got, lse_got, o_want, lse_want, what="", raw=True):
    assert np.all(np.isfinite(o_got)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse_got)), f"{what}: non-finite LSE"
    raw, beyond = o_max_abs(o_got, o_want, raw)
    rl = rel_l2(o_got, o_want)
    ml = max_abs(lse_got, lse_want)
    assert raw <= TOL_O_MAXABS, f"{what}: O max-abs {raw:.3e} (|O_ref| < 2)"
    assert beyond <= TOL_O_MAXABS, f"{what}: O max-abs beyond bf16 storage {beyond:.3e} (|O_ref| >= 2)"
    assert rl <= TOL_O_RELL2, f"{what}: O rel-L2 {rl:.3e}"
    assert ml <= TOL_LSE_MAXABS, f"{what}: LSE max-abs {ml:.3e}"
    return max(raw, beyond), rl, ml


def check_grads(got, want, what=""):
    for name, g, w in zip(("dQ", "dK", "dV"), got, want):
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        rl = rel_l2(g, w)
        assert rl <= TOL_GRAD_RELL2, f"{what}: {name} rel-L2 {rl:.3e}"


def sample_heads(B, H, k, seed=0):
    """k seeded (b, h) pairs, always including the last head."""
    rng = np.random.default_rng(seed)
    total = B * H
    picks = set(rng.choice(total, size=min(k, total), replace=False).tolist())
    picks.add(total - 1)
    return sorted((p // H, p % H) for p in picks)


def sample_rows(N, seed=0, n_mid=256):
    """Rows of the first and last 128-row tiles plus seeded rows in between."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(N, 128))) | set(range(max(0, N - 128), N))
    if N > 256:
        rows |= set(rng.choice(np.arange(128, N - 128), size=min(n_mid, N - 256),
                               replace=False).tolist())
    return np.array(sorted(rows))


def default_scale(d):
    return 1.0 / math.sqrt(d)

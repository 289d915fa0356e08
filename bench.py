#!/usr/bin/env python
"""Attention throughput on one GB300: forward + backward TFLOP/s of the CUDA
kernels behind the C ABI, with the forward and the dK/dV kernel timed on their
own, a roofline figure for the dominant kernel, an end-to-end figure through
host buffers, and the fp64 CPU oracle timed on a bounded sample.

One step = fa_fwd + fa_bwd (all stages) over one batch of seeded synthetic
bf16 inputs. FLOPs: forward 4*B*H*N^2*d (halved when causal), backward 2.5x
that, so a step counts 3.5x the forward FLOPs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--causal] [--impl reference]

Under torchrun (--gpus N > 1) every rank runs an independent replica of the
workload on its own GPU (attention heads are independent; there is no
data-path collective) and rank 0 prints one JSON line: value = all ranks'
FLOPs / the slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd+bwd (bf16, 1 GB300)"

# name -> (B, H, N, d); the GPT-style sweeps keep B*N = 16384 tokens
WORKLOADS = {"b1_h2_n128_d64": (1, 2, 128, 64), "b4_h8_n1024_d64": (4, 8, 1024, 64),
             "long_b1_h16_n32768_d128": (1, 16, 32768, 128)}
for _d, _H in ((64, 32), (128, 16)):
    for _N in (512, 1024, 2048, 4096, 8192, 16384):
        WORKLOADS[f"gpt_d{_d}_n{_N}"] = (16384 // _N, _H, _N, _d)
# the other supported head dims, same token count (hidden 2048 at d = 32)
WORKLOADS["dim_d32_n4096"] = (4, 64, 4096, 32)
WORKLOADS["dim_d96_n4096"] = (4, 16, 4096, 96)
# head dim 256 runs its own forward and dK/dV kernels (fwd256_kernel,
# bwd256_dkdv_kernel)
WORKLOADS["dim_d256_n4096"] = (4, 8, 4096, 256)
DEFAULT_WORKLOAD = "gpt_d128_n4096"

# Packed batches of variable-length sequences (fa_fwd_varlen / fa_bwd_varlen):
# name -> (sequences, H, d, shortest, longest, length seed); the lengths are
# drawn uniformly from [shortest, longest] with the seed, equal for q and k.
VARLEN_WORKLOADS = {"varlen_d128_s16_256to4096": (16, 16, 128, 256, 4096, 7),
                    "varlen_d64_s64_64to1024": (64, 32, 64, 64, 1024, 8)}


# Decode against a key/value cache (fa_decode): name -> (B, H, Nq, Nk, d);
# the cache is [B, Nk, H, d] and sequence b holds a seeded number of valid
# keys in [Nk / 2, Nk] (cache_seqlens). Timed metric: cache bytes read per
# second; one step = one fa_decode call.
DECODE_WORKLOADS = {"decode_b32_h32_nq1_nk8192_d128": (32, 32, 1, 8192, 128),
                    "decode_b1_h32_nq1_nk131072_d128": (1, 32, 1, 131072, 128),
                    "decode_b32_h32_nq4_nk8192_d128": (32, 32, 4, 8192, 128),
                    "decode_b32_h32_nq8_nk8192_d128": (32, 32, 8, 8192, 128),
                    "decode_b32_h32_nq16_nk8192_d128": (32, 32, 16, 8192, 128),
                    "decode_b1_h32_nq8_nk131072_d128": (1, 32, 8, 131072, 128),
                    "decode_b1_h32_nq16_nk131072_d128": (1, 32, 16, 131072, 128)}
DECODE_METRIC = "attention decode: KV-cache GB/s read (bf16, 1 GB300)"


def decode_lengths(name):
    import numpy as np
    B, _, _, Nk, _ = DECODE_WORKLOADS[name]
    return [int(n) for n in np.random.default_rng(9).integers(Nk // 2, Nk + 1, size=B)]


def varlen_lengths(name):
    import numpy as np
    S, _, _, lo, hi, seed = VARLEN_WORKLOADS[name]
    return [int(n) for n in np.random.default_rng(seed).integers(lo, hi + 1, size=S)]

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dK/dV kernel,
# from an ncu capture of the current kernel source (see profiles/), keyed by
# workload and causal flag; None where no capture of the current kernel exists.
# Algorithmic bytes for comparison: q, k, v, dO read and dk, dv written once
# (6 x 64 MiB) plus the fp32 dQ accumulator (128 MiB) = 537 MB at either size.
NCU_TRAFFIC_BYTES: dict = {("gpt_d128_n4096", False): 6.1875e8,
                           ("gpt_d64_n4096", False): 6.2160e8,
                           ("dim_d256_n4096", False): 6.2114e8}


def fwd_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2.0 if causal else f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"burst": float(p["bf16_tflops"]),
                "sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"burst": 1900.0, "sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and self.uuid not in parts[1]:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores (bounded sample)

def oracle_sample(B, H, N, d, causal, seed, budget_s, max_heads, lengths=None):
    """Times oracle forward + backward on whole heads of the workload until
    budget_s has passed (at least one head). With ``lengths`` (a packed batch)
    head b*H + h is sequence b's head h. Returns (TFLOP/s, heads, seconds)."""
    import oracle
    from exact_tiled_attention_28_gb300 import inputs
    scale = 1.0 / math.sqrt(d)
    heads, spent, flops = 0, 0.0, 0.0
    nseq = B if lengths is None else len(lengths)
    while heads < max_heads and (heads == 0 or spent < budget_s):
        b, h = divmod(heads % (nseq * H), H)
        n = N if lengths is None else lengths[b]
        if lengths is None:
            x = inputs.head_inputs_f64(seed, b, h, n, d)
        else:  # the packed generator's block (b, h)
            x = inputs.head_inputs_f64(seed, b, h, n, d, ("q", "do"))
            x.update(inputs.head_inputs_f64(seed + inputs.KV_SEED_OFFSET, b, h, n, d, ("k", "v")))
        t0 = time.perf_counter()
        oracle.head_forward(x["q"], x["k"], x["v"], causal, scale)
        oracle.head_backward(x["q"], x["k"], x["v"], x["do"], causal, scale)
        spent += time.perf_counter() - t0
        flops += 3.5 * fwd_flops(1, 1, n, d, causal)
        heads += 1
    return flops / spent / 1e12, heads, spent


def blas_threads():
    """Threads of the BLAS library numpy's products run on, read from the
    library itself: through threadpoolctl where it is installed, else from the
    OpenBLAS build loaded into this process (its get_num_threads entry point,
    under the names the numpy and scipy-openblas builds export). Returns
    (threads, how) or (None, why)."""
    import numpy as np  # noqa: F401  (loads the BLAS library)
    try:
        import threadpoolctl
        info = [i for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas"]
        if info:
            return max(int(i["num_threads"]) for i in info), "threadpoolctl"
    except Exception:
        pass
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({ln.split()[-1] for ln in f
                            if "openblas" in ln.lower() and ".so" in ln and "/" in ln})
    except OSError:
        paths = []
    for path in paths:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                    "openblas_get_num_threads64_", "openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn()), f"{os.path.basename(path)}:{sym}"
    return None, "no BLAS thread count readable"


def cpu_cores_entry():
    """The cpu_baseline's core count: the BLAS threads numpy used (the
    products); the oracle's elementwise steps run on one thread."""
    n, how = blas_threads()
    if n is None:
        return {"cores": os.cpu_count(), "cores_source": f"os.cpu_count ({how})"}
    return {"cores": n, "cores_source": f"BLAS threads, read from {how}; "
                                        "elementwise numpy steps run on one thread"}


# ---------------------------------------------------------------------------

def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(WORKLOADS) + sorted(VARLEN_WORKLOADS) + sorted(DECODE_WORKLOADS))
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--layout", default="bhnd", choices=("bhnd", "bnhd"),
                    help="memory layout of q, k, v, o, dO and the gradients")
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-legs", action="store_true",
                    help="skip the sustained leg and the extra workloads of the default line")
    ap.add_argument("--dq-path-sweep", action="store_true",
                    help="time the backward's two dQ paths against each other on the GPT-style "
                         "and long-sequence shapes (one JSON line per shape and mask)")
    ap.add_argument("--dq-sweep-shapes", default="",
                    help="comma-separated subset of the dQ path sweep's shapes")
    ap.add_argument("--unit-rates", action="store_true",
                    help="measure the MUFU exp2 and FP32 FMA rates (the softmax's "
                         "secondary roofs) and print them as one JSON line")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def config_of(args, B, H, N, d):
    return {"workload": f"{args.workload}: B={B} H={H} N={N} d={d} "
                        f"{'causal' if args.causal else 'non-causal'} fwd+bwd",
            "B": B, "H": H, "N": N, "d": d, "causal": bool(args.causal),
            "scale": "1/sqrt(d)", "global_batch": B * args.gpus, "seq_len": N,
            "parallelism": f"replicas x{args.gpus}", "layout": args.layout,
            "l2": "inputs larger than L2" if 8 * B * H * N * d * 2 > 129e6 else "L2-resident"}


def run_reference(args):
    """The reference arm: the fp64 oracle as it stands, on the host cores."""
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    if args.workload in DECODE_WORKLOADS:
        B, H, Nq, Nk, d = DECODE_WORKLOADS[args.workload]
        dl = decode_lengths(args.workload)
        for _ in range(args.warmup):
            decode_oracle_sample(B, H, Nq, Nk, d, args.causal, dl, 1000, 0.0, 1)
        nbytes, spent = 0.0, 0.0
        for _ in range(args.steps):
            g, _, sp = decode_oracle_sample(B, H, Nq, Nk, d, args.causal, dl, 1000, 0.0, 1)
            nbytes += g * 1e9 * sp
            spent += sp
        value = nbytes / spent / 1e9
        line = {"impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": spent * 1e3 / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": decode_config_of(args, B, H, Nq, Nk, d, dl),
                "cpu_baseline": {"value": value, "unit": "GB/s", **cpu_cores_entry(),
                                 "kind": "oracle", "sample": "one (sequence, head) block per step"},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    lengths = None
    if args.workload in VARLEN_WORKLOADS:
        S, H, d = VARLEN_WORKLOADS[args.workload][:3]
        lengths = varlen_lengths(args.workload)
        B, N = S, max(lengths)
    else:
        B, H, N, d = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        oracle_sample(B, H, N, d, args.causal, 1000, 0.0, 1, lengths)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):  # each step: the first head of the workload, fwd + bwd
        tf, _, spent = oracle_sample(B, H, N, d, args.causal, 1000, 0.0, 1, lengths)
        flops += tf * 1e12 * spent
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": (config_of(args, B, H, N, d) if lengths is None
                       else varlen_config_of(args, lengths, H, d)),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", **cpu_cores_entry(),
                             "kind": "oracle",
                             "sample": f"one head (first sequence, d={d}) fwd+bwd per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_e2e(fa, torch, host, x0, o0, lse0, dq0, dk0, dv0, ws0, causal, scale, steps,
            compute=None):
    """Times `steps` end-to-end steps (H2D of the inputs, fa_fwd + fa_bwd, D2H of
    every output) with the three stages pipelined across steps. ``compute(xb,
    ob, wb, stream)`` replaces the fa_fwd + fa_bwd pair when given. The copies
    in and the copies out each alternate over two streams: on GB300 the
    host link carries about 205 GB/s in either direction alone and about 280
    GB/s in both at once only with two streams per direction (one per
    direction reached 245). Returns (ms per step, H2D bytes, D2H bytes, H2D
    GB/s alone, D2H GB/s alone)."""
    outs0 = {"o": o0, "lse": lse0, "dq": dq0, "dk": dk0, "dv": dv0}
    bufs = [({n: t for n, t in x0.items()}, outs0, ws0),
            ({n: torch.empty_like(t) for n, t in x0.items()},
             {n: torch.empty_like(t) for n, t in outs0.items()}, torch.empty_like(ws0))]
    out_host = [{n: torch.empty_like(t, device="cpu").pin_memory() for n, t in outs0.items()}
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs0.values())
    s_in = [torch.cuda.Stream(), torch.cuda.Stream()]
    s_out = [torch.cuda.Stream(), torch.cuda.Stream()]
    s_comp = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event()
    in_done = [[ev(), ev()] for _ in range(steps)]
    comp_done = [ev() for _ in range(steps)]
    out_done = [[ev(), ev()] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(s_comp)
    for s in s_in + s_out:
        s.wait_stream(s_comp)
    for k in range(steps):
        xb, ob, wb = bufs[k % 2]
        for c, s in enumerate(s_in):
            with torch.cuda.stream(s):
                if k >= 2:
                    s.wait_event(comp_done[k - 2])  # buffer k % 2 free for new inputs
                for n in list(host)[c::2]:
                    xb[n].copy_(host[n], non_blocking=True)
                in_done[k][c].record(s)
        for c in range(2):
            s_comp.wait_event(in_done[k][c])
        if k >= 2:
            for c in range(2):
                s_comp.wait_event(out_done[k - 2][c])  # outputs k % 2 copied out
        if compute is not None:
            compute(xb, ob, wb, s_comp)
        else:
            fa.fa_fwd(xb["q"], xb["k"], xb["v"], ob["o"], ob["lse"], causal, scale, stream=s_comp)
            fa.fa_bwd(xb["q"], xb["k"], xb["v"], ob["o"], ob["lse"], xb["do"], ob["dq"], ob["dk"],
                      ob["dv"], causal, scale, wb, stream=s_comp)
        comp_done[k].record(s_comp)
        for c, s in enumerate(s_out):
            with torch.cuda.stream(s):
                s.wait_event(comp_done[k])
                for n in list(ob)[c::2]:
                    out_host[k % 2][n].copy_(ob[n], non_blocking=True)
                out_done[k][c].record(s)
    for c in range(2):
        s_comp.wait_event(out_done[steps - 1][c])
    t1.record(s_comp)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps

    def bw(fn, nbytes):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        return nbytes / (a.elapsed_time(b) * 1e-3) / 1e9

    h2d_gbs = bw(lambda: [bufs[0][0][n].copy_(host[n], non_blocking=True) for n in host], h2d)
    d2h_gbs = bw(lambda: [out_host[0][n].copy_(t, non_blocking=True) for n, t in outs0.items()], d2h)
    return ms, h2d, d2h, h2d_gbs, d2h_gbs


def varlen_config_of(args, lengths, H, d):
    T = sum(lengths)
    return {"workload": f"{args.workload}: {len(lengths)} packed sequences of "
                        f"{min(lengths)}..{max(lengths)} tokens (T={T}), H={H} d={d} "
                        f"{'causal' if args.causal else 'non-causal'} fwd+bwd",
            "sequences": len(lengths), "total_tokens": T, "max_seqlen": max(lengths),
            "H": H, "d": d, "causal": bool(args.causal), "scale": "1/sqrt(d)",
            "global_batch": len(lengths) * args.gpus, "seq_len": max(lengths),
            "parallelism": f"replicas x{args.gpus}", "layout": "packed [T, H, d]",
            "l2": "inputs larger than L2" if 8 * T * H * d * 2 > 129e6 else "L2-resident"}


def run_varlen(args):
    """One step = fa_fwd_varlen + fa_bwd_varlen over a packed batch of seeded
    variable-length sequences (the same lengths for queries and keys)."""
    import torch

    import exact_tiled_attention_28_gb300 as fa
    from exact_tiled_attention_28_gb300 import inputs, replicas

    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    fa.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    S, H, d = VARLEN_WORKLOADS[args.workload][:3]
    lengths = varlen_lengths(args.workload)
    causal = bool(args.causal)
    scale = 1.0 / math.sqrt(d)
    seed = replicas.replica_seed(1000, rank)
    bits, cu_q, cu_k = inputs.packed_inputs(seed, lengths, lengths, H, d)
    T = int(cu_q[-1])
    host = {n: inputs.bits_to_torch_bf16(b).pin_memory() for n, b in bits.items()}
    x = {n: t.to(dev) for n, t in host.items()}
    cu = torch.tensor(cu_q, dtype=torch.int32, device=dev)
    mx = max(lengths)
    o = torch.empty_like(x["q"])
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_varlen_workspace_size(S, H, T, mx, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def compute(xb, ob, wb, st):
        fa.fa_fwd_varlen(xb["q"], xb["k"], xb["v"], ob["o"], ob["lse"], cu, cu, mx, mx, causal,
                         scale, stream=st)
        fa.fa_bwd_varlen(xb["q"], xb["k"], xb["v"], ob["o"], ob["lse"], xb["do"], ob["dq"],
                         ob["dk"], ob["dv"], cu, cu, mx, mx, causal, scale, wb, stream=st)

    outs = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd_varlen(x["q"], x["k"], x["v"], o, lse, cu, cu, mx, mx, causal, scale)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_bwd_varlen(x["q"], x["k"], x["v"], o, lse, x["do"], dq, dk, dv, cu, cu, mx, mx,
                         causal, scale, ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status reports an error during warm-up")
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status reports an error in the timed region")
    ms_step = t_start.elapsed_time(t_end) / args.steps
    ms_step_max = replicas.max_over_ranks(ms_step, dev)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    e2e_ms, h2d, d2h, h2d_gbs, d2h_gbs = run_e2e(fa, torch, host, x, o, lse, dq, dk, dv, ws,
                                                 causal, scale, args.e2e_steps, compute=compute)
    F = sum(fwd_flops(1, H, n, d, causal) for n in lengths)
    peaks = load_peaks()
    value = replicas.aggregate_throughput(3.5 * F, world, ms_step_max)
    bwd_tf = 2.5 * F / (bwd_ms * 1e-3) / 1e12
    fwd_tf = F / (fwd_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: Q, K, V, dO i.i.d. N(0,1) rounded to bf16, seeded; seeded lengths",
        "config": varlen_config_of(args, lengths, H, d),
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_burst_peak": fwd_tf / peaks["burst"]},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf},
        "roofline": tensor_roofline("fa_bwd_varlen (all stages)", bwd_tf, peaks,
                                    f"2.5 x sum_b 4*H*n_b^2*d{' / 2' if causal else ''} = "
                                    f"{2.5 * F:.4g} FLOP per launch"),
        "roofline_fwd": tensor_roofline("fwd_kernel (packed batch)", fwd_tf, peaks,
                                        f"{F:.4g} FLOP per launch"),
        "e2e": {"value": 3.5 * F / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": "two copy-in streams, compute, two copy-out streams; double-buffered",
                "h2d_gbs_alone": h2d_gbs, "d2h_gbs_alone": d2h_gbs},
        # per step: check + forward, check + pre-pass + dK/dV + dQ convert
        "gpu_launches": 6 * args.steps,
        "clocks": clocks,
    }
    g_ms = replicas.max_over_ranks(graph_step_ms(fa, torch, step, args.steps), dev)
    line["graph"] = {"ms_per_step": g_ms,
                     "fwd_bwd_tflops": replicas.aggregate_throughput(3.5 * F, world, g_ms),
                     "how": "one step captured into a CUDA graph, replayed `steps` times "
                            "after the timed region; same kernels, no per-call host work"}
    if world > 1:
        torch.distributed.barrier()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, heads, spent = oracle_sample(S, H, mx, d, causal, seed, args.cpu_budget_s, 64, lengths)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", **cpu_cores_entry(),
                                "kind": "oracle",
                                "sample": f"{heads} whole (sequence, head) blocks fwd+bwd, "
                                          f"{spent:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def decode_config_of(args, B, H, Nq, Nk, d, lengths):
    return {"workload": f"{args.workload}: B={B} H={H} Nq={Nq} cache Nk={Nk} d={d} "
                        f"(valid keys {min(lengths)}..{max(lengths)} per sequence), "
                        f"{'causal' if args.causal else 'non-causal'}, forward",
            "B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d, "causal": bool(args.causal),
            "scale": "1/sqrt(d)", "global_batch": B * args.gpus, "seq_len": Nk,
            "parallelism": f"replicas x{args.gpus}", "layout": "cache [B, Nk, H, d]",
            "l2": "cache larger than L2" if 2 * sum(lengths) * H * d * 2 > 129e6 else "L2-resident"}


def decode_oracle_sample(B, H, Nq, Nk, d, causal, lengths, seed, budget_s, max_heads):
    """The oracle on whole (sequence, head) blocks; returns (cache GB/s, heads, s)."""
    import oracle
    from exact_tiled_attention_28_gb300 import inputs
    scale = 1.0 / math.sqrt(d)
    heads, spent, nbytes = 0, 0.0, 0
    while heads < max_heads and (heads == 0 or spent < budget_s):
        b, h = divmod(heads % (B * H), H)
        n = lengths[b]
        x = inputs.head_inputs_f64(seed, b, h, Nq, d, ("q",))
        kv = inputs.head_inputs_f64(seed + inputs.KV_SEED_OFFSET, b, h, Nk, d, ("k", "v"))
        t0 = time.perf_counter()
        oracle.head_forward(x["q"], kv["k"][:n], kv["v"][:n], causal, scale)
        spent += time.perf_counter() - t0
        nbytes += 2 * n * d * 2
        heads += 1
    return nbytes / spent / 1e9, heads, spent


def run_decode(args):
    """One step = one fa_decode call over the workload's cache."""
    import torch

    import exact_tiled_attention_28_gb300 as fa
    from exact_tiled_attention_28_gb300 import inputs, replicas

    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    fa.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    B, H, Nq, Nk, d = DECODE_WORKLOADS[args.workload]
    lengths = decode_lengths(args.workload)
    causal = bool(args.causal)
    scale = 1.0 / math.sqrt(d)
    seed = replicas.replica_seed(1000, rank)
    bits = inputs.nqnk_inputs(seed, B, H, Nq, Nk, d)
    # the cache stored as [B, Nk, H, d], passed as [B, H, Nk, d] views
    k = inputs.bits_to_torch_bf16(bits["k"]).to(dev).transpose(1, 2).contiguous().transpose(1, 2)
    v = inputs.bits_to_torch_bf16(bits["v"]).to(dev).transpose(1, 2).contiguous().transpose(1, 2)
    del bits["k"], bits["v"]
    q_host = inputs.bits_to_torch_bf16(bits["q"]).pin_memory()
    q = q_host.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    cs = torch.tensor(lengths, dtype=torch.int32, device=dev)
    ws = torch.empty(max(fa.fa_decode_workspace_size(B, H, Nq, Nk, d), 16), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()

    def step():
        fa.fa_decode(q, k, v, o, lse, causal, scale, cache_seqlens=cs, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status reports an error during warm-up")
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status reports an error in the timed region")
    ms_step = t_start.elapsed_time(t_end) / args.steps
    ms_step_max = replicas.max_over_ranks(ms_step, dev)
    kv_bytes = 2 * sum(lengths) * H * d * 2
    algo_bytes = kv_bytes + 2 * (B * H * Nq * d * 2) + B * H * Nq * 4  # + q, o, lse
    # end to end: each step copies its new query rows in and o, lse out (pinned
    # host memory); the cache stays resident on the device
    o_host = torch.empty_like(o, device="cpu").pin_memory()
    l_host = torch.empty_like(lse, device="cpu").pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(args.e2e_steps, 1)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n_e2e):
        q.copy_(q_host, non_blocking=True)
        step()
        o_host.copy_(o, non_blocking=True)
        l_host.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    peaks = load_peaks()
    gbs = kv_bytes / (ms_step_max * 1e-3) / 1e9 * world
    achieved = algo_bytes / (ms_step * 1e-3) / 1e9
    # the path fa_decode takes (include/fa.h): Nq >= 8 runs the tensor-core
    # forward, over whole caches when the (batch, head) pairs fill the SMs,
    # else with the keys split (d = 64, 128); otherwise the split-key kernel
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    split = B * H < sms and Nk > 128  # more than one key split per (batch, head)
    if Nq >= 8 and B * H >= sms:
        kernel, launches = "fwd_kernel (tensor cores, whole caches)", 2
    elif Nq >= 8 and d in (64, 128) and split:
        kernel, launches = "fwd_kernel (tensor cores, keys split) + decode_combine_kernel", 3
    else:
        kernel, launches = "decode_split_kernel + decode_combine_kernel", 1 + split
    line = {
        "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: q, K, V i.i.d. N(0,1) rounded to bf16, seeded; seeded cache lengths",
        "config": decode_config_of(args, B, H, Nq, Nk, d, lengths),
        "roofline": {"kernel": kernel, "bound": "hbm",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "peak_kind": f"copy bandwidth of {peaks['source']}", "traffic": None,
                     "algorithmic": f"K and V of the valid keys once, q, o, lse: {algo_bytes:.4g} "
                                    f"bytes per call"},
        "tflops": 4.0 * Nq * sum(lengths) * H * d / (ms_step * 1e-3) / 1e12,
        "e2e": {"value": kv_bytes / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4,
                "note": "the cache stays on the device; each step copies q in and o, lse out"},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if world > 1:
        torch.distributed.barrier()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_, heads, spent = decode_oracle_sample(B, H, Nq, Nk, d, causal, lengths, seed,
                                                args.cpu_budget_s, 512)
        line["cpu_baseline"] = {"value": v_, "unit": "GB/s", **cpu_cores_entry(),
                                "kind": "oracle",
                                "sample": f"{heads} whole (sequence, head) blocks, {spent:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# Extra points of the default line, each timed like the headline (fwd and the
# backward's stages with CUDA events): the causal run of the headline
# workload, the GPT-style d = 64 point at N = 4096 (both masks), the
# long-sequence causal config and the small d = 64 config.
SUB_LINES = (("gpt_d128_n4096", True), ("gpt_d64_n4096", False), ("gpt_d64_n4096", True),
             ("long_b1_h16_n32768_d128", True), ("b4_h8_n1024_d64", False),
             ("b4_h8_n1024_d64", True))

# Seconds of back-to-back headline steps for the sustained-peak leg: the
# driver's default run times about 30 ms, where the burst peak applies; the
# sustained peak is measured on a seconds-long loop, so it is compared only
# with a loop of that length.
SUSTAINED_LEG_S = 2.5


class Problem:
    """Device buffers of one dense [B, H, N, d] workload (inputs seeded)."""

    def __init__(self, torch, fa, inputs, dev, seed, B, H, N, d, layout="bhnd", pin=False):
        self.B, self.H, self.N, self.d = B, H, N, d
        bits = inputs.attention_inputs(seed, B, H, N, d)
        host = {n: inputs.bits_to_torch_bf16(b) for n, b in bits.items()}
        if layout == "bnhd":
            # [B, N, H, d] storage, passed as [B, H, N, d] views (strided entry points)
            host = {n: t.transpose(1, 2).contiguous() for n, t in host.items()}
            if pin:
                host = {n: t.pin_memory() for n, t in host.items()}
            host = {n: t.transpose(1, 2) for n, t in host.items()}
            self.x = {n: t.transpose(1, 2).to(dev).transpose(1, 2) for n, t in host.items()}
            new = lambda: torch.empty((B, N, H, d), dtype=torch.bfloat16, device=dev).transpose(1, 2)
        else:
            if pin:
                host = {n: t.pin_memory() for n, t in host.items()}
            self.x = {n: t.to(dev) for n, t in host.items()}
            new = lambda: torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
        self.host = host
        self.o = new()
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = new(), new(), new()
        self.ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
        self.layout = layout

    def step(self, fa, stream, causal, scale, ev=None):
        """fa_fwd + fa_bwd; with ev (6 events): the forward, the backward and
        its three stages (pre-pass, dK/dV, dQ convert) are bracketed."""
        x = self.x
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(x["q"], x["k"], x["v"], self.o, self.lse, causal, scale)
        if ev is not None:
            ev[1].record(stream)
        if self.layout == "bhnd":
            fa.fa_bwd_stages(x["q"], x["k"], x["v"], self.o, self.lse, x["do"], self.dq, self.dk,
                             self.dv, causal, scale, self.ws,
                             events=None if ev is None else ev[2:6])
        else:  # the staged entry points take contiguous tensors: time fa_bwd as a whole
            if ev is not None:
                ev[2].record(stream)
                ev[3].record(stream)
            fa.fa_bwd(x["q"], x["k"], x["v"], self.o, self.lse, x["do"], self.dq, self.dk,
                      self.dv, causal, scale, self.ws)
            if ev is not None:
                ev[4].record(stream)
                ev[5].record(stream)


def event_means(evs):
    """Mean ms of fwd, pre-pass, dK/dV, dQ convert and the whole backward."""
    m = lambda a, b: statistics.mean(e[a].elapsed_time(e[b]) for e in evs)
    return {"fwd_ms": m(0, 1), "pre_ms": m(2, 3), "dkdv_ms": m(3, 4), "dq_ms": m(4, 5),
            "bwd_ms": m(2, 5)}


def kernel_names(d, layout="bhnd"):
    if layout != "bhnd":
        return "fa_bwd (all stages)", "fwd_kernel"
    return ("bwd256_dkdv_kernel" if d == 256 else "bwd_dkdv_kernel",
            "fwd256_kernel" if d == 256 else "fwd_kernel")


def tensor_roofline(kernel, tflops, peaks, flop, traffic=None):
    """A tensor-bound roofline entry against the burst bf16 peak (the timed
    regions here last milliseconds to tens of milliseconds)."""
    return {"kernel": kernel, "bound": "tensor", "achieved": tflops, "peak": peaks["burst"],
            "unit": "TFLOP/s", "frac": tflops / peaks["burst"],
            "peak_kind": f"burst bf16 of {peaks['source']}", "traffic": traffic,
            "algorithmic": flop}


def sub_line(fa, torch, inputs, dev, stream, seed, name, causal, steps, warmup, peaks):
    """Times one extra workload like the headline; returns its summary."""
    B, H, N, d = WORKLOADS[name]
    scale = 1.0 / math.sqrt(d)
    pb = Problem(torch, fa, inputs, dev, seed, B, H, N, d)
    for _ in range(max(warmup, 3)):
        pb.step(fa, stream, causal, scale)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        pb.step(fa, stream, causal, scale, evs[k])
    torch.cuda.synchronize()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError(f"device status reports an error in sub-line {name}")
    t = event_means(evs)
    F = fwd_flops(B, H, N, d, causal)
    fwd_tf = F / (t["fwd_ms"] * 1e-3) / 1e12
    dkdv_tf = 2.5 * F / (t["dkdv_ms"] * 1e-3) / 1e12
    fb_tf = 3.5 * F / ((t["fwd_ms"] + t["bwd_ms"]) * 1e-3) / 1e12
    g_ms = graph_step_ms(fa, torch, lambda: pb.step(fa, torch.cuda.current_stream(), causal,
                                                    scale), steps)
    kd, kf = kernel_names(d)
    del pb
    torch.cuda.empty_cache()
    return {"workload": f"{name}: B={B} H={H} N={N} d={d} "
                        f"{'causal' if causal else 'non-causal'} fwd+bwd",
            "steps": steps, **{k: v for k, v in t.items()},
            "fwd_tflops": fwd_tf, "fwd_frac_of_burst_peak": fwd_tf / peaks["burst"],
            "fwd_bwd_tflops": fb_tf, "fwd_bwd_frac_of_burst_peak": fb_tf / peaks["burst"],
            "graph": {"ms_per_step": g_ms, "fwd_bwd_tflops": 3.5 * F / (g_ms * 1e-3) / 1e12},
            "roofline": tensor_roofline(kd, dkdv_tf, peaks, f"2.5 x 4*B*H*N^2*d"
                                        f"{' / 2' if causal else ''} = {2.5 * F:.4g} FLOP per launch"),
            "roofline_fwd": tensor_roofline(kf, fwd_tf, peaks, f"{F:.4g} FLOP per launch")}


def graph_step_ms(fa, torch, run, steps):
    """One step (run() enqueues fa_fwd + fa_bwd on the current stream)
    captured into a CUDA graph, then replayed `steps` times back to back: the
    step time without the host's per-call work (argument checks, tensor maps,
    launches). Small workloads are bound by that work when launched call by
    call."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status reports an error in the graph replays")
    del g
    return t0.elapsed_time(t1) / steps


def sustained_leg(fa, torch, pb, stream, causal, scale, seconds, uuid, peaks):
    """Back-to-back headline steps for at least `seconds`, with the clocks
    sampled: the throughput a long run settles at, against the sustained peak."""
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    n, wall0 = 0, time.perf_counter()
    while time.perf_counter() - wall0 < seconds:
        for _ in range(50):
            pb.step(fa, stream, causal, scale)
        n += 50
        torch.cuda.synchronize()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1)
    F = fwd_flops(pb.B, pb.H, pb.N, pb.d, causal)
    tf = 3.5 * F * n / (ms * 1e-3) / 1e12
    return {"leg": "sustained: back-to-back fwd+bwd steps of the headline workload",
            "seconds": ms * 1e-3, "steps": n, "fwd_bwd_tflops": tf,
            "frac_of_sustained_peak": tf / peaks["sustained"],
            "peak_kind": f"sustained bf16 of {peaks['source']}", "clocks": clocks}


def run_ours(args):
    import torch

    import exact_tiled_attention_28_gb300 as fa
    from exact_tiled_attention_28_gb300 import inputs, replicas

    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    fa.load()  # raises if the library is missing: there is no fallback
    dev = torch.device("cuda", torch.cuda.current_device())
    B, H, N, d = WORKLOADS[args.workload]
    causal = bool(args.causal)
    scale = 1.0 / math.sqrt(d)
    seed = replicas.replica_seed(1000, rank)
    pb = Problem(torch, fa, inputs, dev, seed, B, H, N, d, layout=args.layout, pin=True)
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 3)):
        pb.step(fa, stream, causal, scale)
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status reports a timeout during warm-up")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(args.steps):
        pb.step(fa, stream, causal, scale, evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    if fa.fa_last_device_status() != fa.FA_OK:
        raise RuntimeError("device status reports a timeout in the timed region")
    ms_total = t_start.elapsed_time(t_end)
    t = event_means(evs)
    ms_step = ms_total / args.steps

    ms_step_max = replicas.max_over_ranks(ms_step, dev)

    # end to end through host buffers: every step copies its inputs in from
    # pinned host memory and all of its outputs back. Copies in, compute and
    # copies out run on three streams with double-buffered device tensors, so
    # step k+1's inputs arrive while step k computes and step k-1's outputs leave.
    e2e_ms, h2d, d2h, h2d_gbs, d2h_gbs = run_e2e(fa, torch, pb.host, pb.x, pb.o, pb.lse, pb.dq,
                                                 pb.dk, pb.dv, pb.ws, causal, scale,
                                                 args.e2e_steps)

    F = fwd_flops(B, H, N, d, causal)
    peaks = load_peaks()
    value = replicas.aggregate_throughput(3.5 * F, world, ms_step_max)
    dkdv_tf = 2.5 * F / (t["dkdv_ms"] * 1e-3) / 1e12
    fwd_tf = F / (t["fwd_ms"] * 1e-3) / 1e12
    fb_tf = 3.5 * F / ((t["fwd_ms"] + t["bwd_ms"]) * 1e-3) / 1e12
    traffic = NCU_TRAFFIC_BYTES.get((args.workload, causal)) if args.layout == "bhnd" else None
    kd, kf = kernel_names(d, args.layout)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: Q, K, V, dO i.i.d. N(0,1) rounded to bf16, seeded",
        "config": config_of(args, B, H, N, d),
        "fwd": {"ms": t["fwd_ms"], "tflops": fwd_tf,
                "frac_of_burst_peak": fwd_tf / peaks["burst"]},
        "fwd_bwd": {"tflops": fb_tf, "frac_of_burst_peak": fb_tf / peaks["burst"]},
        "bwd": {"ms": t["bwd_ms"], "pre_ms": t["pre_ms"], "dkdv_ms": t["dkdv_ms"],
                "dq_ms": t["dq_ms"], "tflops": 2.5 * F / (t["bwd_ms"] * 1e-3) / 1e12},
        "roofline": tensor_roofline(kd, dkdv_tf, peaks,
                                    f"2.5 x 4*B*H*N^2*d{' / 2' if causal else ''} = "
                                    f"{2.5 * F:.4g} FLOP per launch", traffic),
        "roofline_fwd": tensor_roofline(kf, fwd_tf, peaks, f"{F:.4g} FLOP per launch"),
        "e2e": {"value": 3.5 * F / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": "two copy-in streams, compute, two copy-out streams; double-buffered",
                "h2d_gbs_alone": h2d_gbs, "d2h_gbs_alone": d2h_gbs},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    if args.layout == "bhnd":
        g_ms = replicas.max_over_ranks(
            graph_step_ms(fa, torch, lambda: pb.step(fa, torch.cuda.current_stream(), causal,
                                                     scale), args.steps), dev)
        line["graph"] = {"ms_per_step": g_ms,
                         "fwd_bwd_tflops": replicas.aggregate_throughput(3.5 * F, world, g_ms),
                         "how": "one step captured into a CUDA graph, replayed `steps` times "
                                "after the timed region; same kernels, no per-call host work"}
    if not args.no_extra_legs and args.layout == "bhnd":
        line["sustained"] = sustained_leg(fa, torch, pb, stream, causal, scale,
                                          SUSTAINED_LEG_S, uuid, peaks)
        if args.workload == DEFAULT_WORKLOAD and not causal:
            del pb
            torch.cuda.empty_cache()
            line["sub_lines"] = [sub_line(fa, torch, inputs, dev, stream, seed, name, c,
                                          min(args.steps, 20), args.warmup, peaks)
                                 for name, c in SUB_LINES]
    if world > 1:
        torch.distributed.barrier()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, heads, spent = oracle_sample(B, H, N, d, causal, seed, args.cpu_budget_s, 64)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", **cpu_cores_entry(),
                                "kind": "oracle",
                                "sample": f"{heads} whole heads (N={N}, d={d}) fwd+bwd, "
                                          f"{spent:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# The two dQ paths of the backward timed against each other (the atomic
# accumulation inside the dK/dV kernel, and the dK/dV kernel without dQ plus
# the query-stationary dQ kernel): name -> (B, H, N, d).
DQ_SWEEP = {"gpt_d128_n4096": (4, 16, 4096, 128), "gpt_d128_n8192": (2, 16, 8192, 128),
            "long_b1_h16_n32768_d128": (1, 16, 32768, 128), "gpt_d64_n4096": (4, 32, 4096, 64),
            "gpt_d64_n8192": (2, 32, 8192, 64), "b1_h32_n32768_d64": (1, 32, 32768, 64)}


def run_dq_path_sweep(args):
    """One JSON line per (shape, mask): fa_bwd_with_dq_path timed with CUDA
    events on each dQ path (warm-up, then --steps calls each, alternating)."""
    import torch

    import exact_tiled_attention_28_gb300 as fa
    from exact_tiled_attention_28_gb300 import inputs
    torch.cuda.set_device(0)
    fa.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    shapes = args.dq_sweep_shapes.split(",") if args.dq_sweep_shapes else list(DQ_SWEEP)
    for name in shapes:
        B, H, N, d = DQ_SWEEP[name]
        scale = 1.0 / math.sqrt(d)
        pb = Problem(torch, fa, inputs, dev, 1000, B, H, N, d)
        x = pb.x
        for causal in (False, True):
            fa.fa_fwd(x["q"], x["k"], x["v"], pb.o, pb.lse, causal, scale)

            def bwd(path):
                fa.fa_bwd(x["q"], x["k"], x["v"], pb.o, pb.lse, x["do"], pb.dq, pb.dk, pb.dv,
                          causal, scale, pb.ws, dq_path=path)

            paths = (fa.FA_DQ_ATOMIC, fa.FA_DQ_SEPARATE)
            for _ in range(max(args.warmup, 3)):
                for p in paths:
                    bwd(p)
            ms = {p: [] for p in paths}
            for _ in range(args.steps):
                for p in paths:
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    bwd(p)
                    e1.record(stream)
                    ms[p].append((e0, e1))
            torch.cuda.synchronize()
            if fa.fa_last_device_status() != fa.FA_OK:
                raise RuntimeError(f"device status reports an error in {name}")
            F = 2.5 * fwd_flops(B, H, N, d, causal)
            out = {}
            for p, label in ((fa.FA_DQ_ATOMIC, "atomic"), (fa.FA_DQ_SEPARATE, "separate")):
                t = statistics.median(a.elapsed_time(b) for a, b in ms[p])
                out[label] = {"bwd_ms": t, "bwd_tflops": F / (t * 1e-3) / 1e12,
                              "frac_of_burst_peak": F / (t * 1e-3) / 1e12 / peaks["burst"]}
            print(json.dumps({"dq_path_sweep": f"{name}: B={B} H={H} N={N} d={d} "
                                               f"{'causal' if causal else 'non-causal'}",
                              "steps": args.steps, **out,
                              "separate_over_atomic": out["separate"]["bwd_ms"] /
                                                      out["atomic"]["bwd_ms"]}), flush=True)
        del pb
        torch.cuda.empty_cache()


def run_unit_rates(args):
    """The secondary roofs next to the tensor pipe: MUFU exp2 and FP32 FMA
    operations per clock per SM, and the bf16 tensor rate per SM for
    comparison (the measured burst peak over the SM count and its clock)."""
    import torch

    import exact_tiled_attention_28_gb300 as fa
    torch.cuda.set_device(0)
    fa.load()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(0).uuid)
    except Exception:
        pass
    fa.fa_measure_unit_rates(256)  # warm-up
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    r = fa.fa_measure_unit_rates(8192)
    clocks = sampler.stop()
    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = clocks.get("sm_mhz") or 2070.0
    tensor_flop_per_clk_sm = peaks["burst"] * 1e12 / sms / (mhz * 1e6)
    # per score: the forward's two products cost 4 d FLOPs and its softmax one
    # exp2; the ratio bounds how far the exponentials may fall behind
    r.update({"unit": "operations per clock per SM", "sms": sms, "clocks": clocks,
              "tensor_bf16_flop_per_clk_per_sm_burst": tensor_flop_per_clk_sm,
              "scores_per_clk_per_sm_tensor_d128": tensor_flop_per_clk_sm / (4 * 128),
              "scores_per_clk_per_sm_tensor_d64": tensor_flop_per_clk_sm / (4 * 64)})
    print(json.dumps(r), flush=True)


def main():
    args = parse_args()
    if args.unit_rates:
        run_unit_rates(args)
        return
    if args.dq_path_sweep:
        run_dq_path_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in VARLEN_WORKLOADS:
        run_varlen(args)
    elif args.workload in DECODE_WORKLOADS:
        run_decode(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

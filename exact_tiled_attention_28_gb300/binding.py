"""ctypes binding of libfa.so (the C ABI in include/fa.h).

Argument marshalling only: every step of the attention computation runs in
the library's CUDA kernels. There is no fallback of any kind; if the library
is missing or fails to load, every call raises.

The tensor-level helpers take ``torch`` CUDA tensors (PyTorch provides device
memory and streams here, nothing else) and pass their raw device pointers,
sizes and the current CUDA stream to the C functions of the same names.
"""

from __future__ import annotations

import ctypes
import os

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_WORKSPACE = 5
FA_ERR_DEVICE_CHECK = 6

# every symbol include/fa.h declares
EXPORTED = ("fa_abi_version", "fa_fwd", "fa_fwd_strided", "fa_bwd_workspace_size", "fa_bwd",
            "fa_bwd_strided", "fa_bwd_preprocess",
            "fa_bwd_dkdv", "fa_bwd_dq_finalize", "fa_bwd_noalloc", "fa_bwd_with_dq_path", "fa_selftest_wait_timeout",
            "fa_set_wait_limit_ns", "fa_is_debug_build", "fa_selftest_index_check",
            "fa_selftest_exp2",
            "fa_status_string", "fa_last_device_status", "fa_fwd_nqnk", "fa_bwd_nqnk",
            "fa_fwd_varlen", "fa_bwd_varlen_workspace_size", "fa_bwd_varlen",
            "fa_decode_workspace_size", "fa_decode", "fa_measure_unit_rates")

# dq_path of fa_bwd_with_dq_path
FA_DQ_AUTO, FA_DQ_ATOMIC, FA_DQ_SEPARATE = 0, 1, 2

# fixed device scratch of fa_bwd_noalloc (FA_NOALLOC_SCRATCH_BYTES in include/fa.h)
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
# default limit of the kernels' bounded waits (FA_WAIT_LIMIT_NS_DEFAULT)
WAIT_LIMIT_NS_DEFAULT = 2_000_000_000

_lib = None      # the library every call below goes through
_loaded = {}     # debug flag -> loaded library


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string_safe(status)}")


def library_path(debug: bool = False) -> str:
    """libfa.so, or with debug=True the debug build libfa_debug.so (index
    checks on every store, settable wait limit; include/fa.h)."""
    name = "libfa_debug.so" if debug else "libfa.so"
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), name)


def use_library(debug: bool):
    """Routes every later call through the release (False) or the debug (True)
    library; returns the one used before, as a debug flag."""
    global _lib
    before = _lib is not None and _lib is _loaded.get(True)
    _lib = _load_path(bool(debug))
    return before


def load():
    """Loads libfa.so (once) and declares the C signatures. Raises if absent."""
    global _lib
    if _lib is None:
        _lib = _load_path(False)
    return _lib


def _load_path(debug: bool):
    if debug in _loaded:
        return _loaded[debug]
    path = library_path(debug)
    if not os.path.exists(path):
        raise FaError(FA_ERR_CUDA, f"{path} is not built; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_abi_version.restype = i
    lib.fa_abi_version.argtypes = []
    lib.fa_fwd.restype = i
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    ll = ctypes.POINTER(ctypes.c_longlong)
    lib.fa_fwd_strided.restype = i
    lib.fa_fwd_strided.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ll, i, f, vp]
    lib.fa_bwd_strided.restype = i
    lib.fa_bwd_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, ll, i, f, vp,
                                   sz, vp]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.fa_bwd_preprocess.restype = i
    lib.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, vp, sz, vp]
    lib.fa_bwd_dkdv.restype = i
    lib.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.fa_bwd_dq_finalize.restype = i
    lib.fa_bwd_dq_finalize.argtypes = [vp, i, i, i, i, f, vp, sz, vp]
    lib.fa_bwd_with_dq_path.restype = i
    lib.fa_bwd_with_dq_path.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.fa_selftest_exp2.restype = i
    lib.fa_selftest_exp2.argtypes = [vp, vp, i, vp]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [i, vp]
    lib.fa_set_wait_limit_ns.restype = i
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_is_debug_build.restype = i
    lib.fa_is_debug_build.argtypes = []
    lib.fa_selftest_index_check.restype = i
    lib.fa_selftest_index_check.argtypes = [vp]
    lib.fa_measure_unit_rates.restype = i
    lib.fa_measure_unit_rates.argtypes = [vp, i, vp]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [i]
    lib.fa_last_device_status.restype = i
    lib.fa_last_device_status.argtypes = [vp]
    lib.fa_fwd_nqnk.restype = i
    lib.fa_fwd_nqnk.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ll, i, f, vp]
    lib.fa_bwd_nqnk.restype = i
    lib.fa_bwd_nqnk.argtypes = [vp] * 9 + [i, i, i, i, i, ll, i, f, vp, sz, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_fwd_varlen.argtypes = [vp] * 7 + [i] * 7 + [ll, i, f, vp]
    lib.fa_bwd_varlen_workspace_size.restype = sz
    lib.fa_bwd_varlen_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_bwd_varlen.restype = i
    lib.fa_bwd_varlen.argtypes = [vp] * 11 + [i] * 7 + [ll, i, f, vp, sz, vp]
    lib.fa_decode_workspace_size.restype = sz
    lib.fa_decode_workspace_size.argtypes = [i] * 5
    lib.fa_decode.restype = i
    lib.fa_decode.argtypes = [vp] * 6 + [i] * 5 + [ll, i, f, vp, sz, vp]
    _loaded[debug] = lib
    return lib


def status_string_safe(status: int) -> str:
    try:
        return load().fa_status_string(int(status)).decode()
    except Exception:  # the library itself failed to load
        return f"status {status}"


def fa_status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FaError(status, where)


def _stream_handle(stream) -> int:
    """cudaStream_t of `stream`, or of the current device's current stream.
    PyTorch's raw getter returns the same handle as
    torch.cuda.current_stream().cuda_stream without building a Stream object
    (0.1 against 2.9 us per call on the GB300 host), which matters when small
    problems are launched call by call."""
    import torch
    if stream is not None:
        return int(stream.cuda_stream)
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return int(raw(torch.cuda.current_device()))
    return int(torch.cuda.current_stream().cuda_stream)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def _dev_ptr(t, name, dtype, shape, strided=False):
    """Device pointer of a tensor. With strided=True any view of that shape
    whose last dimension is contiguous is accepted; otherwise the tensor must
    be contiguous."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}")
    if strided:
        if t.stride(-1) != 1 and t.shape[-1] > 1:
            raise ValueError(f"{name}: the last dimension must be contiguous")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check_workspace(workspace):
    import torch
    if not workspace.is_cuda or workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")


def _strides(tensors):
    """ctypes array of (batch, head, row) element strides of [B, H, N, d] views,
    or None when every view is contiguous."""
    if all(t.is_contiguous() for t in tensors):
        return None
    vals = []
    for t in tensors:
        vals += [int(t.stride(0)), int(t.stride(1)), int(t.stride(2))]
    return (ctypes.c_longlong * len(vals))(*vals)


# ---------------------------------------------------------------------------
# raw-pointer calls (the C ABI as is)

def fa_fwd_raw(q, k, v, o, lse, B, H, N, d, causal, scale, stream) -> int:
    return load().fa_fwd(q, k, v, o, lse, B, H, N, d, int(bool(causal)), float(scale), stream)


def fa_bwd_raw(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, causal, scale, workspace,
               workspace_bytes, stream) -> int:
    return load().fa_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, int(bool(causal)),
                         float(scale), workspace, workspace_bytes, stream)


def fa_bwd_preprocess_raw(o, lse, do, B, H, N, d, workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd_preprocess(o, lse, do, B, H, N, d, workspace, workspace_bytes, stream)


def fa_bwd_dkdv_raw(q, k, v, do, dk, dv, B, H, N, d, causal, scale, workspace, workspace_bytes,
                    stream) -> int:
    return load().fa_bwd_dkdv(q, k, v, do, dk, dv, B, H, N, d, int(bool(causal)), float(scale),
                              workspace, workspace_bytes, stream)


def fa_bwd_dq_finalize_raw(dq, B, H, N, d, scale, workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd_dq_finalize(dq, B, H, N, d, float(scale), workspace, workspace_bytes,
                                     stream)


def fa_bwd_noalloc_raw(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, causal, scale,
                       stream) -> int:
    return load().fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, int(bool(causal)),
                                 float(scale), stream)


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, d))


def fa_measure_unit_rates(iters: int = 4096) -> dict:
    """Runs the arithmetic-unit microbenchmark on the current device and
    returns operations per clock per SM for the MUFU exp2 (ex2.approx), FFMA
    and the two-lane FFMA2 (counted in FMAs), with the cycle counts. Waits for
    the device (a measurement, not a step of the attention path)."""
    import torch
    cyc = torch.zeros(6, dtype=torch.int64, device="cuda")
    _check(load().fa_measure_unit_rates(cyc.data_ptr(), int(iters), _stream_handle(None)),
           "fa_measure_unit_rates")
    torch.cuda.synchronize()
    c = [int(x) for x in cyc.cpu()]
    ops = 2 * 1024 * 8 * int(iters)  # per SM, per kernel
    return {"ex2_per_clk_per_sm": ops / c[0], "ffma_per_clk_per_sm": ops / c[2],
            "ffma2_fma_per_clk_per_sm": 2 * ops / c[4], "cycles": [c[0], c[2], c[4]],
            "iters": int(iters)}


def fa_selftest_wait_timeout(limit_ms: int, stream=None) -> None:
    _check(load().fa_selftest_wait_timeout(int(limit_ms), _stream_handle(stream)),
           "fa_selftest_wait_timeout")


def fa_set_wait_limit_ns(limit_ns: int) -> None:
    """Debug build: the limit of every bounded on-chip wait of the kernels (0 =
    give up at once when a wait does not complete at its first try)."""
    _check(load().fa_set_wait_limit_ns(int(limit_ns)), "fa_set_wait_limit_ns")


def fa_is_debug_build() -> bool:
    return bool(load().fa_is_debug_build())


def fa_selftest_index_check(stream=None) -> None:
    """Debug build: a kernel whose one index check fails (no memory access)."""
    _check(load().fa_selftest_index_check(_stream_handle(stream)), "fa_selftest_index_check")


def fa_selftest_exp2(x, y, stream=None) -> None:
    """y <- 2^x with the forward kernel's FMA-pipe exponential (CUDA fp32 tensors)."""
    import torch
    n = x.numel()
    _dev_ptr(x, "x", torch.float32, x.shape)
    _dev_ptr(y, "y", torch.float32, x.shape)
    _check(load().fa_selftest_exp2(x.data_ptr(), y.data_ptr(), n, _stream_handle(stream)),
           "fa_selftest_exp2")


def fa_last_device_status(stream=None) -> int:
    return int(load().fa_last_device_status(_stream_handle(stream)))


# ---------------------------------------------------------------------------
# tensor-level calls

def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """o, lse <- attention(q, k, v) on the current (or given) CUDA stream.

    q, o are [B, H, Nq, d] and k, v [B, H, Nk, d] bf16 views with a contiguous
    last dimension (a [B, N, H, d] tensor passed as .transpose(1, 2), or K and
    V slices of one packed buffer, go through the strided entry points); lse
    is contiguous fp32 [B, H, Nq]. Nq != Nk goes through fa_fwd_nqnk (causal
    mask aligned at the bottom right)."""
    import torch
    B, H, N, d = _shape(q)
    Nk = int(k.shape[2]) if k.dim() == 4 else -1
    bf = torch.bfloat16
    ts = ((q, "q"), (k, "k"), (v, "v"), (o, "o"))
    args = [_dev_ptr(t, n, bf, (B, H, Nk if n in ("k", "v") else N, d), strided=True)
            for t, n in ts]
    args.append(_dev_ptr(lse, "lse", torch.float32, (B, H, N)))
    st = _strides([t for t, _ in ts])
    if Nk != N:
        _check(load().fa_fwd_nqnk(*args, B, H, N, Nk, d, st, int(bool(causal)), float(scale),
                                  _stream_handle(stream)), "fa_fwd_nqnk")
    elif st is None:
        _check(fa_fwd_raw(*args, B, H, N, d, causal, scale, _stream_handle(stream)), "fa_fwd")
    else:
        _check(load().fa_fwd_strided(*args, B, H, N, d, st, int(bool(causal)), float(scale),
                                     _stream_handle(stream)), "fa_fwd_strided")


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float, workspace,
           stream=None, dq_path=None) -> None:
    """dq, dk, dv <- gradients of sum(o * do); workspace is a CUDA uint8 tensor of at
    least fa_bwd_workspace_size(B, H, Nq, d) bytes. Shapes as for fa_fwd (dk, dv
    like k, dq and do like q). dq_path (FA_DQ_ATOMIC, FA_DQ_SEPARATE or
    FA_DQ_AUTO) goes through fa_bwd_with_dq_path; it takes contiguous
    [B, H, N, d] tensors of equal query and key lengths."""
    import torch
    B, H, N, d = _shape(q)
    Nk = int(k.shape[2]) if k.dim() == 4 else -1
    bf = torch.bfloat16
    ts = ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do"), (dq, "dq"), (dk, "dk"), (dv, "dv"))
    p = {n: _dev_ptr(t, n, bf, (B, H, Nk if n in ("k", "v", "dk", "dv") else N, d), strided=True)
         for t, n in ts}
    pl = _dev_ptr(lse, "lse", torch.float32, (B, H, N))
    _check_workspace(workspace)
    ptrs = [p["q"], p["k"], p["v"], p["o"], pl, p["do"], p["dq"], p["dk"], p["dv"]]
    st = _strides([t for t, _ in ts])
    if dq_path is not None:
        if Nk != N or st is not None:
            raise ValueError("dq_path takes contiguous [B, H, N, d] tensors of one length N")
        _check(load().fa_bwd_with_dq_path(*ptrs, B, H, N, d, int(bool(causal)), float(scale),
                                          int(dq_path), workspace.data_ptr(), workspace.numel(),
                                          _stream_handle(stream)), "fa_bwd_with_dq_path")
    elif Nk != N:
        _check(load().fa_bwd_nqnk(*ptrs, B, H, N, Nk, d, st, int(bool(causal)), float(scale),
                                  workspace.data_ptr(), workspace.numel(),
                                  _stream_handle(stream)), "fa_bwd_nqnk")
    elif st is None:
        _check(fa_bwd_raw(*ptrs, B, H, N, d, causal, scale, workspace.data_ptr(),
                          workspace.numel(), _stream_handle(stream)), "fa_bwd")
    else:
        _check(load().fa_bwd_strided(*ptrs, B, H, N, d, st, int(bool(causal)), float(scale),
                                     workspace.data_ptr(), workspace.numel(),
                                     _stream_handle(stream)), "fa_bwd_strided")


def fa_bwd_stages(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float, workspace,
                  stream=None, events=None) -> None:
    """fa_bwd as its three C-ABI stages. If ``events`` is a list of four CUDA
    events, they are recorded before, between and after the stages (the
    benchmark times the dK/dV stage with them)."""
    import torch
    B, H, N, d = _shape(q)
    bf = torch.bfloat16
    shp = (B, H, N, d)
    P = {n: _dev_ptr(t, n, bf, shp) for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"),
                                                  (do, "do"), (dq, "dq"), (dk, "dk"), (dv, "dv"))}
    pl = _dev_ptr(lse, "lse", torch.float32, (B, H, N))
    ws, nws = workspace.data_ptr(), workspace.numel()
    st = _stream_handle(stream)
    s = None
    if events:
        s = torch.cuda.current_stream() if stream is None else stream
        events[0].record(s)
    _check(fa_bwd_preprocess_raw(P["o"], pl, P["do"], B, H, N, d, ws, nws, st), "fa_bwd_preprocess")
    if events:
        events[1].record(s)
    _check(fa_bwd_dkdv_raw(P["q"], P["k"], P["v"], P["do"], P["dk"], P["dv"], B, H, N, d, causal,
                           scale, ws, nws, st), "fa_bwd_dkdv")
    if events:
        events[2].record(s)
    _check(fa_bwd_dq_finalize_raw(P["dq"], B, H, N, d, scale, ws, nws, st), "fa_bwd_dq_finalize")
    if events:
        events[3].record(s)


def fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float,
                   stream=None) -> None:
    """fa_bwd without a workspace argument: the library's fixed device scratch
    array is used, nothing is allocated. For callers that cannot allocate
    device memory; sizes whose workspace exceeds NOALLOC_SCRATCH_BYTES raise
    (FA_ERR_WORKSPACE). Calls overlapping on the GPU race on the shared array."""
    import torch
    B, H, N, d = _shape(q)
    bf = torch.bfloat16
    ptrs = [_dev_ptr(t, n, bf, (B, H, N, d))
            for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"))]
    ptrs.append(_dev_ptr(lse, "lse", torch.float32, (B, H, N)))
    ptrs += [_dev_ptr(t, n, bf, (B, H, N, d))
             for t, n in ((do, "do"), (dq, "dq"), (dk, "dk"), (dv, "dv"))]
    _check(fa_bwd_noalloc_raw(*ptrs, B, H, N, d, causal, scale, _stream_handle(stream)),
           "fa_bwd_noalloc")


# ---------------------------------------------------------------------------
# packed batches of variable-length sequences

def fa_bwd_varlen_workspace_size(B: int, H: int, total_q: int, max_seqlen_k: int, d: int) -> int:
    return int(load().fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_k, d))


def _varlen_args(q, k, v, tensors_q, tensors_k, cu_seqlens_q, cu_seqlens_k):
    """Pointers, sizes and (head, row) strides of packed [T, H, d] views."""
    import torch
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("expected packed [T, H, d] tensors")
    Tq, H, d = (int(x) for x in q.shape)
    Tk = int(k.shape[0])
    bf = torch.bfloat16
    ptrs = {}
    for t, n in tensors_q:
        ptrs[n] = _dev_ptr(t, n, bf, (Tq, H, d), strided=True)
    for t, n in tensors_k:
        ptrs[n] = _dev_ptr(t, n, bf, (Tk, H, d), strided=True)
    B = int(cu_seqlens_q.numel()) - 1
    for c, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _dev_ptr(c, n, torch.int32, (B + 1,))
    order = list(tensors_q[:1]) + list(tensors_k) + list(tensors_q[1:])
    return Tq, Tk, H, d, B, ptrs, order


def _varlen_strides(tensors):
    if all(t.is_contiguous() for t in tensors):
        return None
    vals = []
    for t in tensors:
        vals += [int(t.stride(1)), int(t.stride(0))]
    return (ctypes.c_longlong * len(vals))(*vals)


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, causal: bool, scale: float, stream=None) -> None:
    """o, lse <- attention of a packed batch: q, o [total_q, H, d] and k, v
    [total_k, H, d] bf16 views with a contiguous last dimension; cu_seqlens_q,
    cu_seqlens_k int32 CUDA tensors of B + 1 prefix offsets; lse fp32
    [H, total_q]. Causal masks are aligned at the bottom right per sequence."""
    import torch
    Tq, Tk, H, d, B, p, _ = _varlen_args(q, k, v, ((q, "q"), (o, "o")), ((k, "k"), (v, "v")),
                                         cu_seqlens_q, cu_seqlens_k)
    pl = _dev_ptr(lse, "lse", torch.float32, (H, Tq))
    st = _varlen_strides([q, k, v, o])
    _check(load().fa_fwd_varlen(p["q"], p["k"], p["v"], p["o"], pl, cu_seqlens_q.data_ptr(),
                                cu_seqlens_k.data_ptr(), B, H, Tq, Tk, int(max_seqlen_q),
                                int(max_seqlen_k), d, st, int(bool(causal)), float(scale),
                                _stream_handle(stream)), "fa_fwd_varlen")


def fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu_seqlens_q, cu_seqlens_k,
                  max_seqlen_q: int, max_seqlen_k: int, causal: bool, scale: float, workspace,
                  stream=None) -> None:
    """dq, dk, dv <- gradients of sum(o * do) for a packed batch (see
    fa_fwd_varlen); workspace is a CUDA uint8 tensor of at least
    fa_bwd_varlen_workspace_size(B, H, total_q, max_seqlen_k, d) bytes."""
    import torch
    Tq, Tk, H, d, B, p, _ = _varlen_args(
        q, k, v, ((q, "q"), (o, "o"), (do, "do"), (dq, "dq")),
        ((k, "k"), (v, "v"), (dk, "dk"), (dv, "dv")), cu_seqlens_q, cu_seqlens_k)
    pl = _dev_ptr(lse, "lse", torch.float32, (H, Tq))
    _check_workspace(workspace)
    st = _varlen_strides([q, k, v, o, do, dq, dk, dv])
    _check(load().fa_bwd_varlen(p["q"], p["k"], p["v"], p["o"], pl, p["do"], p["dq"], p["dk"],
                                p["dv"], cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, H,
                                Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), d, st,
                                int(bool(causal)), float(scale), workspace.data_ptr(),
                                workspace.numel(), _stream_handle(stream)), "fa_bwd_varlen")


# ---------------------------------------------------------------------------
# decode against a key/value cache

def fa_decode_workspace_size(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().fa_decode_workspace_size(B, H, Nq, Nk, d))


def fa_decode(q, k_cache, v_cache, o, lse, causal: bool, scale: float, cache_seqlens=None,
              workspace=None, stream=None) -> None:
    """o, lse <- attention of Nq <= 16 new rows per (batch, head) against the
    cache: q, o [B, H, Nq, d] and k_cache, v_cache [B, H, Nk, d] bf16 views
    with a contiguous last dimension (a [B, Nk, H, d] cache passed as
    .transpose(1, 2) is fine); lse fp32 [B, H, Nq]; cache_seqlens an int32
    CUDA tensor of B valid key counts, or None; workspace a CUDA uint8 tensor
    of fa_decode_workspace_size(...) bytes."""
    import torch
    B, H, Nq, d = _shape(q)
    Nk = int(k_cache.shape[2]) if k_cache.dim() == 4 else -1
    bf = torch.bfloat16
    ts = ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (o, "o"))
    ptrs = [_dev_ptr(t, n, bf, (B, H, Nk if n.endswith("cache") else Nq, d), strided=True)
            for t, n in ts]
    pl = _dev_ptr(lse, "lse", torch.float32, (B, H, Nq))
    cs = 0
    if cache_seqlens is not None:
        cs = _dev_ptr(cache_seqlens, "cache_seqlens", torch.int32, (B,))
    wp, wn = 0, 0
    if workspace is not None:
        _check_workspace(workspace)
        wp, wn = workspace.data_ptr(), workspace.numel()
    st = _strides([t for t, _ in ts])
    _check(load().fa_decode(*ptrs, pl, cs or None, B, H, Nq, Nk, d, st, int(bool(causal)),
                            float(scale), wp or None, wn, _stream_handle(stream)), "fa_decode")

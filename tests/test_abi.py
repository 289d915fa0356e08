"""The C ABI on the host: the library loads, exports every function that
include/fa.h declares, and rejects bad arguments before launching anything.
No call here reaches a GPU."""

import ctypes
import os
import re

import pytest

import exact_tiled_attention_28_gb300 as fa
from exact_tiled_attention_28_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.library_path()):
        from exact_tiled_attention_28_gb300 import build
        build.build()
    return fa.load()


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(fa_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    decl = declared_functions()
    assert "fa_fwd" in decl and "fa_bwd" in decl
    for name in decl:
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert set(decl) <= set(binding.EXPORTED)


def test_abi_version(lib):
    assert lib.fa_abi_version() == 2


def test_status_strings(lib):
    for code in range(7):
        s = fa.fa_status_string(code)
        assert s.startswith("FA_")
    assert "unknown" in fa.fa_status_string(99)


P = 4096  # a 16-byte-aligned fake address: never dereferenced, the calls fail first


def fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return binding.fa_fwd_raw(q, k, v, o, lse, B, H, N, d, causal, scale, None)


def bwd(lib, ws=P, ws_bytes=None, B=1, H=1, N=128, d=64, scale=0.125, null=None):
    ptrs = [P] * 9
    if null is not None:
        ptrs[null] = None
    if ws_bytes is None:
        ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    return binding.fa_bwd_raw(*ptrs, B, H, N, d, 0, scale, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=P + 8), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=80), fa.FA_ERR_UNSUPPORTED),
    (dict(d=48), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(B=65536, H=32768), fa.FA_ERR_UNSUPPORTED),
])
def test_fwd_rejects_before_launch(lib, kw, want):
    assert fwd(lib, **kw) == want


def test_bwd_rejects_before_launch(lib):
    for i in range(9):
        assert bwd(lib, null=i) == fa.FA_ERR_INVALID_ARG
    assert bwd(lib, d=48) == fa.FA_ERR_UNSUPPORTED
    assert bwd(lib, d=512) == fa.FA_ERR_UNSUPPORTED
    assert bwd(lib, ws=None) == fa.FA_ERR_WORKSPACE
    assert bwd(lib, ws=P + 4) == fa.FA_ERR_WORKSPACE
    assert bwd(lib, ws_bytes=fa.fa_bwd_workspace_size(1, 1, 128, 64) - 1) == fa.FA_ERR_WORKSPACE


def test_workspace_size(lib):
    for B, H, N, d in ((1, 1, 1, 64), (4, 8, 1024, 64), (1, 16, 32768, 128), (2, 3, 77, 128),
                       (2, 2, 100, 32), (1, 3, 300, 96)):
        assert fa.fa_bwd_workspace_size(B, H, N, d) >= 4 * B * H * N * (d + 1)
    assert fa.fa_bwd_workspace_size(1, 1, 0, 64) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 16, 80) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: without the shared library every call raises."""
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_loaded", {})
    monkeypatch.setattr(binding, "library_path",
                        lambda debug=False: str(tmp_path / "libfa.so"))
    with pytest.raises(fa.FaError):
        binding.load()
    with pytest.raises(fa.FaError):
        fa.fa_bwd_workspace_size(1, 1, 128, 64)
    with pytest.raises(fa.FaError):
        binding.use_library(True)


def test_debug_build_exports_the_same_symbols(lib):
    """libfa_debug.so (FA_DEBUG: index checks, settable wait limit) has every
    declared entry point; only it honours the debug hooks."""
    dbg = binding._load_path(True)
    for name in declared_functions():
        assert hasattr(dbg, name), f"{name} not exported by the debug build"
    assert dbg.fa_is_debug_build() == 1 and lib.fa_is_debug_build() == 0
    assert lib.fa_set_wait_limit_ns(0) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_selftest_index_check(None) == fa.FA_ERR_UNSUPPORTED
    # the debug build checks the limit before any device call
    assert dbg.fa_set_wait_limit_ns(binding.WAIT_LIMIT_NS_DEFAULT + 1) == fa.FA_ERR_INVALID_ARG
    before = binding.use_library(True)
    try:
        assert fa.fa_is_debug_build()
    finally:
        binding.use_library(before)
    assert not fa.fa_is_debug_build()


def test_dq_path_rejects_before_launch(lib):
    def call(path, d=64):
        return lib.fa_bwd_with_dq_path(*([P] * 9), 1, 2, 256, d, 0, 0.125, path, P,
                                       fa.fa_bwd_workspace_size(1, 2, 256, d), None)
    assert call(3) == fa.FA_ERR_INVALID_ARG
    assert call(-1) == fa.FA_ERR_INVALID_ARG
    for d in (32, 96, 256):  # the separate dQ kernel takes d = 64 and 128
        assert call(fa.FA_DQ_SEPARATE, d) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd_with_dq_path(*([P] * 8), None, 1, 2, 256, 64, 0, 0.125, 2, P,
                                   fa.fa_bwd_workspace_size(1, 2, 256, 64), None) == \
        fa.FA_ERR_INVALID_ARG


def test_library_has_no_torch_dependency(lib):
    """The C ABI takes plain pointers: the shared object links no torch library."""
    path = fa.library_path()
    data = open(path, "rb").read()
    assert b"libtorch" not in data and b"libc10" not in data
    assert isinstance(lib, ctypes.CDLL)


def test_exp2_selftest_rejects_before_launch(lib):
    assert lib.fa_selftest_exp2(None, P, 4, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_exp2(P, P, 0, None) == fa.FA_ERR_INVALID_ARG


def test_strided_entry_points_reject_bad_strides(lib):
    import ctypes
    good = [4 * 8 * 64, 8 * 64, 64] * 8
    for bad in (0, -8, 12, 1 << 36):
        st = list(good)
        st[4] = bad
        arr = (ctypes.c_longlong * 24)(*st)
        assert lib.fa_fwd_strided(P, P, P, P, P, 1, 4, 8, 64, arr, 0, 0.125, None) == \
            fa.FA_ERR_INVALID_ARG
        assert lib.fa_bwd_strided(*([P] * 9), 1, 4, 8, 64, arr, 0, 0.125, P, 1 << 20, None) == \
            fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_strided(P, P, P, P, P, 1, 4, 8, 64, None, 0, 0.125, None) == \
        fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_strided(*([P] * 9), 1, 4, 8, 64, None, 0, 0.125, P, 1 << 20, None) == \
        fa.FA_ERR_INVALID_ARG


def test_nqnk_entry_points_reject_before_launch(lib):
    def fwd(q=P, B=1, H=2, Nq=100, Nk=300, d=64, st=None, scale=0.125):
        return lib.fa_fwd_nqnk(q, P, P, P, P, B, H, Nq, Nk, d, st, 1, scale, None)

    assert fwd(q=None) == fa.FA_ERR_INVALID_ARG
    assert fwd(Nk=0) == fa.FA_ERR_INVALID_ARG
    assert fwd(Nq=0) == fa.FA_ERR_INVALID_ARG
    assert fwd(d=80) == fa.FA_ERR_UNSUPPORTED
    assert fwd(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    bad = (ctypes.c_longlong * 12)(*([64 * 300 * 2, 64 * 300, 64] * 3 + [64, 0, 64]))
    assert fwd(st=bad) == fa.FA_ERR_INVALID_ARG
    ws_ok = fa.fa_bwd_workspace_size(1, 2, 100, 64)
    assert lib.fa_bwd_nqnk(*([P] * 9), 1, 2, 100, 300, 64, None, 1, 0.125, P, ws_ok - 1,
                           None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd_nqnk(*([P] * 8), None, 1, 2, 100, 300, 64, None, 1, 0.125, P, ws_ok,
                           None) == fa.FA_ERR_INVALID_ARG


def test_varlen_entry_points_reject_before_launch(lib):
    def fwd(cu_q=P, cu_k=P, B=3, H=2, Tq=500, Tk=700, mq=300, mk=400, d=128, st=None):
        return lib.fa_fwd_varlen(P, P, P, P, P, cu_q, cu_k, B, H, Tq, Tk, mq, mk, d, st, 1,
                                 0.1, None)

    assert fwd(cu_q=None) == fa.FA_ERR_INVALID_ARG
    assert fwd(cu_k=P + 2) == fa.FA_ERR_INVALID_ARG
    for kw in (dict(Tk=0), dict(mq=0), dict(mk=0), dict(B=0), dict(Tq=0)):
        assert fwd(**kw) == fa.FA_ERR_INVALID_ARG, kw
    assert fwd(d=256) == fa.FA_ERR_UNSUPPORTED
    assert fwd(B=1 << 20, H=1 << 11, mq=1 << 10) == fa.FA_ERR_UNSUPPORTED
    assert fwd(st=(ctypes.c_longlong * 8)(128, 256, 128, 256, 128, 256, 128, 12)) == \
        fa.FA_ERR_INVALID_ARG
    ws = fa.fa_bwd_varlen_workspace_size(3, 2, 500, 400, 128)
    # D and lse2 padded per sequence, plus the fp32 accumulator
    assert ws >= 4 * (2 * 2 * (512 + 128 * 4) + 2 * 500 * 128)
    assert fa.fa_bwd_varlen_workspace_size(3, 2, 500, 400, 48) == 0
    assert fa.fa_bwd_varlen_workspace_size(3, 2, 500, 0, 128) == 0
    assert lib.fa_bwd_varlen(*([P] * 11), 3, 2, 500, 700, 300, 400, 128, None, 0, 0.1, P, ws - 1,
                             None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_bwd_varlen(*([P] * 11), 3, 2, 500, 700, 300, 400, 128, None, 0, 0.1, None, ws,
                             None) == fa.FA_ERR_WORKSPACE


def test_decode_rejects_before_launch(lib):
    def dec(q=P, cs=None, B=2, H=4, Nq=1, Nk=1000, d=128, st=None, scale=0.1):
        return lib.fa_decode(q, P, P, P, P, cs, B, H, Nq, Nk, d, st, 1, scale, None, 0, None)

    assert dec(q=None) == fa.FA_ERR_INVALID_ARG
    assert dec(Nq=17) == fa.FA_ERR_UNSUPPORTED
    assert dec(Nq=0) == fa.FA_ERR_INVALID_ARG
    assert dec(Nk=0) == fa.FA_ERR_INVALID_ARG
    assert dec(d=80) == fa.FA_ERR_UNSUPPORTED
    assert dec(cs=P + 2) == fa.FA_ERR_INVALID_ARG
    assert dec(scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert dec(st=(ctypes.c_longlong * 12)(*([64] * 11 + [3]))) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_decode_workspace_size(1, 1, 1, 1 << 17, 128) >= 152 * (128 + 1) * 4
    assert fa.fa_decode_workspace_size(1, 1, 17, 1000, 128) == 0


def test_d256_dense_forward_and_backward_only(lib):
    """d = 256 passes the dense forward's and backward's argument checks (on a
    host without a GPU the call then fails at the device query, not as
    unsupported); the unequal-length, packed and decode entry points reject
    it."""
    assert fwd(lib, d=256) != fa.FA_ERR_UNSUPPORTED
    assert fwd(lib, d=256, q=None) == fa.FA_ERR_INVALID_ARG
    ws = fa.fa_bwd_workspace_size(1, 1, 128, 256)
    # D and lse2 rows (2 x 128 fp32) and the fp32 dQ accumulator (128 x 256)
    assert ws == (2 * 128 + 128 * 256) * 4
    assert bwd(lib, d=256, ws_bytes=ws) != fa.FA_ERR_UNSUPPORTED
    assert bwd(lib, d=256, ws_bytes=ws) != fa.FA_ERR_INVALID_ARG
    assert bwd(lib, d=256, ws_bytes=ws - 1) == fa.FA_ERR_WORKSPACE
    assert bwd(lib, d=256, null=3, ws_bytes=ws) == fa.FA_ERR_INVALID_ARG
    # 64-key work items are counted in int
    assert fa.fa_bwd_workspace_size(1 << 15, 1 << 10, 1 << 12, 256) == 0
    assert lib.fa_fwd_nqnk(P, P, P, P, P, 1, 1, 10, 20, 256, None, 0, 0.1, None) == \
        fa.FA_ERR_UNSUPPORTED
    assert lib.fa_decode(P, P, P, P, P, None, 1, 1, 1, 100, 256, None, 0, 0.1, None, 0, None) == \
        fa.FA_ERR_UNSUPPORTED


def test_unit_rates_rejects_before_launch(lib):
    assert lib.fa_measure_unit_rates(None, 16, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_measure_unit_rates(P + 4, 16, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_measure_unit_rates(P, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_measure_unit_rates(P, (1 << 20) + 1, None) == fa.FA_ERR_INVALID_ARG

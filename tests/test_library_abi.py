"""CPU checks of the C ABI: the library loads, exports every entry point that
include/fa.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

from tiled_online_softmax_sm_gb300 import binding as fb
from tiled_online_softmax_sm_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fb.load()


def _declared():
    with open(os.path.join(ROOT, "include", "fa.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_documented_entry_points():
    assert _declared() == sorted(fb.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def _fwd(lib, **kw):
    args = dict(q=16, k=16, v=16, o=16, lse=16, B=1, H=2, Hkv=1, n=8, m=8, d=128, dv=128,
                scale=0.1, causal=0)
    args.update(kw)
    return lib.fa_forward(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                          args["H"], args["Hkv"], args["n"], args["m"], args["d"], args["dv"],
                          args["scale"], args["causal"], None)


def test_forward_validation(lib):
    assert _fwd(lib, H=3, Hkv=2) == fb.FA_ERR_INVALID_ARG
    assert _fwd(lib, n=-1) == fb.FA_ERR_INVALID_ARG
    assert _fwd(lib, q=None) == fb.FA_ERR_INVALID_ARG
    assert _fwd(lib, q=8) == fb.FA_ERR_INVALID_ARG        # misaligned
    assert _fwd(lib, causal=2) == fb.FA_ERR_INVALID_ARG
    assert _fwd(lib, d=96, dv=96) == fb.FA_ERR_UNSUPPORTED
    assert _fwd(lib, d=128, dv=64) == fb.FA_ERR_UNSUPPORTED
    assert _fwd(lib, scale=0.0) == fb.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=-1.0) == fb.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=0) == fb.FA_OK                     # nothing to do: no launch
    assert _fwd(lib, n=0) == fb.FA_OK


def test_dense_size_limits(lib):
    # token rows b*n + i and the LSE stride H*n are 32-bit in the kernels
    big = 1 << 30
    assert lib.fa_forward(16, 16, 16, 16, 16, 2, 1, 1, big, 1, 128, 128, 0.1, 0, None) == \
        fb.FA_ERR_UNSUPPORTED
    assert lib.fa_forward(16, 16, 16, 16, 16, 1, 2, 2, big, 1, 64, 64, 0.1, 0, None) == \
        fb.FA_ERR_UNSUPPORTED
    assert lib.fa_forward(16, 16, 16, 16, 16, 2, 1, 1, 1, big, 128, 128, 0.1, 0, None) == \
        fb.FA_ERR_UNSUPPORTED
    assert lib.fa_forward_fp8(16, 16, 16, 16, 16, 2, 1, 1, big, 1, 128, 128, 0.1, 1.0, 1.0, 1.0,
                              0, None) == fb.FA_ERR_UNSUPPORTED
    assert lib.fa_forward_f32(16, 16, 16, 16, 16, 1, 65536, 1, 8, 8, 64, 64, 0.1, 0, None) == \
        fb.FA_ERR_UNSUPPORTED
    assert lib.fa_forward_f32(16, 16, 16, 16, 16, 65536, 1, 1, 8, 8, 64, 64, 0.1, 0, None) == \
        fb.FA_ERR_UNSUPPORTED


def test_forward_f32_and_varlen_validation(lib):
    assert lib.fa_forward_f32(16, 16, 16, 16, 16, 1, 4, 3, 8, 8, 64, 64, 0.1, 0, None) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_forward_f32(16, 16, 16, 16, 16, 1, 4, 2, 8, 8, 32, 64, 0.1, 0, None) == fb.FA_ERR_UNSUPPORTED
    assert lib.fa_forward_varlen(16, 16, 16, 16, 16, None, None, 2, 10, 10, 8, 8, 4, 4, 64, 64,
                                 0.1, 1, None) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_forward_varlen(16, 16, 16, 16, 16, 16, 16, 2, 10, 10, 8, 8, 4, 4, 64, 128, 0.1,
                                 1, None) == fb.FA_ERR_UNSUPPORTED
    assert lib.fa_forward_varlen(16, 16, 16, 16, 16, 16, 16, 2, -1, 10, 8, 8, 4, 4, 64, 64, 0.1,
                                 1, None) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_forward_varlen(16, 16, 16, 16, 16, 16, 16, 0, 0, 0, 0, 0, 4, 4, 64, 64, 0.1, 1,
                                 None) == fb.FA_OK


@pytest.mark.parametrize("scale", [0.0, -0.125, float("inf"), float("nan")])
def test_every_forward_and_decode_refuses_a_scale_that_is_not_positive_and_finite(lib, scale):
    """Every entry point that takes a softmax scale requires it positive and
    finite ("手搓 Attention" §1 and §4: the scale is 1/sqrt(d) and the row
    maximum is taken on scaled scores, which for the fp32 kernel's unscaled
    maximum only holds for a positive scale)."""
    assert _fwd(lib, scale=scale) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_forward_f32(16, 16, 16, 16, 16, 1, 2, 1, 8, 8, 64, 64, scale, 0, None) == \
        fb.FA_ERR_INVALID_ARG
    assert lib.fa_forward_fp8(16, 16, 16, 16, 16, 1, 2, 1, 8, 8, 128, 128, scale, 1.0, 1.0, 1.0, 0,
                              None) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_forward_varlen(16, 16, 16, 16, 16, 16, 16, 2, 10, 10, 8, 8, 4, 4, 64, 64, scale,
                                 1, None) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_paged_prefill(16, 16, 16, 16, 16, 16, 16, 16, 2, 10, 8, 4, 4, 64, 64, 16, 100, 8,
                                scale, 1, None) == fb.FA_ERR_INVALID_ARG
    assert _dec(lib, scale=scale) == fb.FA_ERR_INVALID_ARG
    assert _noalloc(lib, scale=scale) == fb.FA_ERR_INVALID_ARG
    assert "scale" in fb.fa_last_error()


def test_decode_workspace_size(lib):
    S, H, dv, X = 64, 32, 128, 16
    tri = S * H * X
    r = lambda x: (x + 255) // 256 * 256
    # the fused form's ticket words, then partial m, l, o
    assert fb.fa_paged_decode_workspace_size(S, H, dv, X) == \
        r(S * H * 4) + 2 * r(tri * 4) + r(tri * dv * 4)
    assert fb.fa_paged_decode_workspace_size(0, H, dv, X) == 0
    assert fb.fa_paged_decode_workspace_size(S, 0, dv, X) == 0


def _dec(lib, **kw):
    a = dict(q=16, kc=16, vc=16, bt=16, sl=16, o=16, lse=16, S=4, H=32, Hkv=8, d=128, dv=128,
             page=16, P=100, maxb=8, X=4, scale=0.1, ws=256, wsb=1 << 20)
    a.update(kw)
    return lib.fa_paged_decode(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["o"], a["lse"], a["S"],
                               a["H"], a["Hkv"], a["d"], a["dv"], a["page"], a["P"], a["maxb"],
                               a["X"], a["scale"], a["ws"], a["wsb"], None)


def test_decode_validation(lib):
    assert _dec(lib, X=0) == fb.FA_ERR_INVALID_ARG
    assert _dec(lib, X=65) == fb.FA_ERR_INVALID_ARG
    assert _dec(lib, H=30) == fb.FA_ERR_INVALID_ARG
    assert _dec(lib, page=32) == fb.FA_ERR_UNSUPPORTED
    assert _dec(lib, d=64, dv=64) == fb.FA_ERR_UNSUPPORTED
    assert _dec(lib, H=64, Hkv=2) == fb.FA_ERR_UNSUPPORTED       # group of 32 > 16
    assert _dec(lib, ws=None) == fb.FA_ERR_WORKSPACE
    assert _dec(lib, wsb=100) == fb.FA_ERR_WORKSPACE
    assert _dec(lib, ws=272) == fb.FA_ERR_WORKSPACE            # not 256-byte aligned
    assert _dec(lib, bt=None) == fb.FA_ERR_INVALID_ARG
    assert _dec(lib, S=0) == fb.FA_OK
    # 32-bit page rows and unit counts
    assert _dec(lib, P=1 << 25) == fb.FA_ERR_UNSUPPORTED
    assert _dec(lib, S=1 << 26, X=64) == fb.FA_ERR_UNSUPPORTED


def test_fused_decode_validation(lib):
    """fa_paged_decode_fused checks its arguments exactly as fa_paged_decode."""
    def fused(**kw):
        a = dict(q=16, kc=16, vc=16, bt=16, sl=16, o=16, lse=16, S=4, H=32, Hkv=8, d=128, dv=128,
                 page=16, P=100, maxb=8, X=4, scale=0.1, ws=256, wsb=1 << 20)
        a.update(kw)
        return lib.fa_paged_decode_fused(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["o"],
                                         a["lse"], a["S"], a["H"], a["Hkv"], a["d"], a["dv"],
                                         a["page"], a["P"], a["maxb"], a["X"], a["scale"], a["ws"],
                                         a["wsb"], None)
    for kw in (dict(X=0), dict(X=65), dict(H=30), dict(page=32), dict(d=64, dv=64),
               dict(H=64, Hkv=2), dict(ws=None), dict(wsb=100), dict(ws=272), dict(bt=None),
               dict(P=1 << 25), dict(S=1 << 26, X=64), dict(scale=0.0), dict(scale=float("nan"))):
        assert fused(**kw) == _dec(lib, **kw), kw
        assert fused(**kw) != fb.FA_OK, kw
    assert fused(S=0) == fb.FA_OK


def _noalloc(lib, **kw):
    a = dict(q=16, kc=16, vc=16, bt=16, sl=16, o=16, lse=16, S=4, H=32, Hkv=8, d=128, dv=128,
             page=16, P=100, maxb=8, X=4, scale=0.1)
    a.update(kw)
    return lib.fa_paged_decode_noalloc(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["o"], a["lse"],
                                       a["S"], a["H"], a["Hkv"], a["d"], a["dv"], a["page"], a["P"],
                                       a["maxb"], a["X"], a["scale"], None)


def test_noalloc_decode_validation(lib):
    """The allocation-free decode checks its arguments as fa_paged_decode
    does, before any launch (and before its first-call address lookup)."""
    assert _noalloc(lib, X=0) == fb.FA_ERR_INVALID_ARG
    assert _noalloc(lib, H=30) == fb.FA_ERR_INVALID_ARG
    assert _noalloc(lib, page=32) == fb.FA_ERR_UNSUPPORTED
    assert _noalloc(lib, d=64, dv=64) == fb.FA_ERR_UNSUPPORTED
    assert _noalloc(lib, bt=None) == fb.FA_ERR_INVALID_ARG
    assert _noalloc(lib, q=24) == fb.FA_ERR_INVALID_ARG          # not 16-byte aligned
    assert _noalloc(lib, S=0) == fb.FA_OK
    # 32-bit page rows (page * Hkv + head) * 16
    assert _noalloc(lib, P=1 << 25) == fb.FA_ERR_UNSUPPORTED


def _gather(lib, **kw):
    a = dict(kc=16, vc=16, bt=16, sl=16, ko=16, vo=16, S=4, Hkv=8, d=128, page=16, P=100, maxb=8,
             X=4)
    a.update(kw)
    return lib.fa_paged_gather(a["kc"], a["vc"], a["bt"], a["sl"], a["ko"], a["vo"], a["S"],
                               a["Hkv"], a["d"], a["page"], a["P"], a["maxb"], a["X"], None)


def test_gather_validation(lib):
    assert _gather(lib, X=0) == fb.FA_ERR_INVALID_ARG
    assert _gather(lib, X=65) == fb.FA_ERR_INVALID_ARG
    assert _gather(lib, Hkv=0) == fb.FA_ERR_INVALID_ARG
    assert _gather(lib, S=-1) == fb.FA_ERR_INVALID_ARG
    assert _gather(lib, d=64) == fb.FA_ERR_UNSUPPORTED
    assert _gather(lib, page=32) == fb.FA_ERR_UNSUPPORTED
    assert _gather(lib, ko=None) == fb.FA_ERR_INVALID_ARG
    assert _gather(lib, vo=24) == fb.FA_ERR_INVALID_ARG          # not 16-byte aligned
    assert _gather(lib, P=0) == fb.FA_ERR_INVALID_ARG
    assert _gather(lib, S=0) == fb.FA_OK
    assert _gather(lib, P=1 << 25) == fb.FA_ERR_UNSUPPORTED
    assert _gather(lib, S=1 << 26, X=64) == fb.FA_ERR_UNSUPPORTED


def test_combine_validation(lib):
    assert lib.fa_split_combine(16, 16, 16, 16, 16, 4, 8, 0, 128, None) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_split_combine(16, 16, 16, 16, 16, 4, 8, 4, 130, None) == fb.FA_ERR_UNSUPPORTED
    assert lib.fa_split_combine(None, 16, 16, 16, 16, 4, 8, 4, 128, None) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_split_combine(16, 16, 16, 16, 16, 0, 8, 4, 128, None) == fb.FA_OK
    assert lib.fa_split_combine(16, 16, 16, 16, 16, 1 << 27, 32, 4, 128, None) == \
        fb.FA_ERR_UNSUPPORTED


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(fb.FaError):
        fb._lib_saved = fb._lib
        try:
            fb._lib = None
            fb.load(str(tmp_path / "nope.so"))
        finally:
            fb._lib = fb._lib_saved

"""Float64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline call it; the CUDA library never does, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain loops, double precision, OpenMP
over query rows); this module only compiles it and marshals numpy arrays.
Each wrapper names the passage it follows; the readings taken where the pages
are silent are listed at the top of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP, -O2).

    No -ffast-math: IEEE double semantics are part of the oracle.
    """
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_attention_rows_f64.argtypes = [P, P, P, I, I, I, I, I, I, I, D, I, P, I, P, P, P]
            lib.oracle_attention_f64.argtypes = [P, P, P, I, I, I, I, I, I, I, D, I, P, P]
            lib.oracle_varlen_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, D, I, P, P]
            lib.oracle_paged_decode_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, D, P, P]
            lib.oracle_paged_prefill_f64.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, D, I, P, P]
            lib.oracle_decode_partials_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, D, P, P, P]
            lib.oracle_split_combine_f64.argtypes = [P, P, P, I, I, I, I, P, P]
            lib.oracle_online_recurrence_f64.argtypes = [P, P, P, I, I, I, I, D, I, I, I, P, P, P]
            lib.oracle_set_num_threads.argtypes = [I]
            for f in ("oracle_attention_rows_f64", "oracle_attention_f64", "oracle_varlen_f64",
                      "oracle_paged_decode_f64", "oracle_paged_prefill_f64",
                      "oracle_decode_partials_f64",
                      "oracle_split_combine_f64", "oracle_online_recurrence_f64",
                      "oracle_num_threads", "oracle_set_num_threads"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc == -2:
        raise IndexError(f"{what}: block-table id out of range")
    if rc != 0:
        raise ValueError(f"{what}: invalid arguments (rc={rc})")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Threads the following oracle calls use; returns the previous count.
    Results do not depend on it (each row is one thread's loop)."""
    return int(_load().oracle_set_num_threads(int(n)))


def attention(q, k, v, scale, causal=False):
    """Dense attention, every row ("手搓 Attention" §2 version 0 + §4).

    q [B,n,H,d], k [B,m,Hkv,d], v [B,m,Hkv,dv] -> (o [B,n,H,dv], lse [B,H,n]), float64.
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, n, H, d = q.shape
    _, m, Hkv, dv = v.shape
    assert k.shape == (B, m, Hkv, d), (k.shape, (B, m, Hkv, d))
    o = np.empty((B, n, H, dv), np.float64)
    lse = np.empty((B, H, n), np.float64)
    rc = _load().oracle_attention_f64(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, n, m, d, dv,
                                      float(scale), int(bool(causal)), _ptr(o), _ptr(lse))
    _check(rc, "oracle.attention")
    return o, lse


def attention_rows(q, k, v, scale, causal, rows, with_weights=False):
    """Selected rows of dense attention; rows is an int array [R,3] of (b, h, i).

    Returns (o [R,dv], lse [R]) and, with with_weights, the softmax weights
    [R,m] (zero for invisible keys): the instrumented mode.
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    rows = _i32(rows).reshape(-1, 3)
    B, n, H, d = q.shape
    _, m, Hkv, dv = v.shape
    R = rows.shape[0]
    o = np.empty((R, dv), np.float64)
    lse = np.empty((R,), np.float64)
    w = np.empty((R, m), np.float64) if with_weights else None
    rc = _load().oracle_attention_rows_f64(
        _ptr(q), _ptr(k), _ptr(v), B, H, Hkv, n, m, d, dv, float(scale), int(bool(causal)),
        _ptr(rows), R, _ptr(o), _ptr(lse), _ptr(w) if w is not None else None)
    _check(rc, "oracle.attention_rows")
    return (o, lse, w) if with_weights else (o, lse)


def varlen(q, k, v, cu_q, cu_k, scale, causal=False):
    """Packed variable-length attention. q [Tq,H,d], k [Tk,Hkv,d], v [Tk,Hkv,dv].

    Returns (o [Tq,H,dv], lse [H,Tq]).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    cu_q, cu_k = _i32(cu_q), _i32(cu_k)
    Tq, H, d = q.shape
    _, Hkv, dv = v.shape
    S = cu_q.shape[0] - 1
    o = np.empty((Tq, H, dv), np.float64)
    lse = np.empty((H, Tq), np.float64)
    rc = _load().oracle_varlen_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_q), _ptr(cu_k), S, H, Hkv,
                                   d, dv, float(scale), int(bool(causal)), _ptr(o), _ptr(lse))
    _check(rc, "oracle.varlen")
    return o, lse


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, scale):
    """Paged single-token decode ("S12 FlashAttention", 实现).

    q [S,H,d]; k_cache [P,Hkv,page,d]; v_cache [P,Hkv,page,dv];
    block_table [S,max_blocks] int; seq_lens [S] int -> (o [S,H,dv], lse [S,H]).
    """
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    bt, sl = _i32(block_table), _i32(seq_lens)
    S, H, d = q.shape
    P, Hkv, page, dv = vc.shape
    o = np.empty((S, H, dv), np.float64)
    lse = np.empty((S, H), np.float64)
    rc = _load().oracle_paged_decode_f64(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(sl), S, H,
                                         Hkv, d, dv, page, P, bt.shape[1], float(scale),
                                         _ptr(o), _ptr(lse))
    _check(rc, "oracle.paged_decode")
    return o, lse


def paged_prefill(q, cu_q, k_cache, v_cache, block_table, seq_lens, scale, causal=True):
    """Several query tokens per sequence against its paged keys.

    q [Tq,H,d] packed by cu_q [S+1]; caches [P,Hkv,page,d]; block_table
    [S,max_blocks]; seq_lens [S] keys per sequence -> (o [Tq,H,dv], lse [H,Tq]).
    Causal: the queries are the last n_s of the seq_lens[s] positions.
    """
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    cu, bt, sl = _i32(cu_q), _i32(block_table), _i32(seq_lens)
    Tq, H, d = q.shape
    P, Hkv, page, dv = vc.shape
    S = cu.shape[0] - 1
    o = np.empty((Tq, H, dv), np.float64)
    lse = np.empty((H, Tq), np.float64)
    rc = _load().oracle_paged_prefill_f64(_ptr(q), _ptr(cu), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(sl),
                                          S, H, Hkv, d, dv, page, P, bt.shape[1], float(scale),
                                          int(bool(causal)), _ptr(o), _ptr(lse))
    _check(rc, "oracle.paged_prefill")
    return o, lse


def decode_partials(q, k_cache, v_cache, block_table, seq_lens, num_splits, scale):
    """Per-split (m, l, o) triples of flash-decoding ("S12 FlashAttention", 练习 1).

    Returns part_m [S,H,X], part_l [S,H,X], part_o [S,H,X,dv].
    """
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    bt, sl = _i32(block_table), _i32(seq_lens)
    S, H, d = q.shape
    P, Hkv, page, dv = vc.shape
    X = int(num_splits)
    pm = np.empty((S, H, X), np.float64)
    pl = np.empty((S, H, X), np.float64)
    po = np.empty((S, H, X, dv), np.float64)
    rc = _load().oracle_decode_partials_f64(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(sl), S, H,
                                            Hkv, d, dv, page, P, bt.shape[1], X, float(scale),
                                            _ptr(pm), _ptr(pl), _ptr(po))
    _check(rc, "oracle.decode_partials")
    return pm, pl, po


def split_combine(part_m, part_l, part_o):
    """Merge (m, l, o) triples with the recurrence's rescale rule.

    part_m, part_l [S,H,X]; part_o [S,H,X,dv] -> (o [S,H,dv], lse [S,H]).
    """
    pm, pl, po = _f64(part_m), _f64(part_l), _f64(part_o)
    S, H, X, dv = po.shape
    o = np.empty((S, H, dv), np.float64)
    lse = np.empty((S, H), np.float64)
    rc = _load().oracle_split_combine_f64(_ptr(pm), _ptr(pl), _ptr(po), S, H, X, dv,
                                          _ptr(o), _ptr(lse))
    _check(rc, "oracle.split_combine")
    return o, lse


def online_recurrence(q, k, v, scale, causal=False, q_block=64, kv_block=64, kv_order=None):
    """The tiled online-softmax recurrence, single head, in double.

    q [n,d], k [m,d], v [m,dv] -> (o [n,dv], lse [n]).  kv_order permutes the
    order in which kv blocks are visited (e.g. diagonal block first).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    n, d = q.shape
    m, dv = v.shape
    order = _i32(kv_order) if kv_order is not None else None
    o = np.empty((n, dv), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().oracle_online_recurrence_f64(
        _ptr(q), _ptr(k), _ptr(v), n, m, d, dv, float(scale), int(bool(causal)),
        int(q_block), int(kv_block), _ptr(order) if order is not None else None,
        _ptr(o), _ptr(lse))
    _check(rc, "oracle.online_recurrence")
    return o, lse

"""ctypes binding of libfa_gb300.so (the C ABI of include/fa.h).

Argument marshalling only: every function here converts its arguments to
pointers and ints and calls the entry point of the same name; all the
arithmetic runs in the library's CUDA kernels.  Pointer arguments may be torch
tensors (their data_ptr is passed), plain ints, or None.  A non-zero status
raises FaError with the library's message.  There is no fallback: if the
library is missing or cannot be loaded, the first call raises.

The helpers at the end (``forward``, ``forward_f32``, ``forward_varlen``,
``paged_decode``, ``paged_decode_fused``, ``split_combine``) allocate outputs
with torch and then call the same entry points.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# FA_LIBRARY selects another build of the same ABI (the debug build,
# libfa_gb300_debug.so, for instance); by default the in-tree library.
LIB_PATH = os.environ.get("FA_LIBRARY") or os.path.join(HERE, "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_WORKSPACE = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5
FA_ERR_BAD_BLOCK_TABLE = 6
FA_ERR_DEBUG_CHECK = 7

EXPORTED = ("fa_forward", "fa_forward_fp8", "fa_forward_f32", "fa_forward_varlen", "fa_paged_prefill",
            "fa_paged_decode_workspace_size",
            "fa_paged_decode", "fa_paged_decode_fused", "fa_paged_decode_noalloc", "fa_paged_gather", "fa_split_combine",
            "fa_last_error",
            "fa_get_device_status")
FA_NOALLOC_SCRATCH_BYTES = 16 << 20


class FaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"fa status {status}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise FaError(FA_ERR_UNSUPPORTED,
                          f"{path} is missing: build it with tiled_online_softmax_sm_gb300.build")
        lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_forward.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
        lib.fa_forward_f32.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
        lib.fa_forward_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, F, F, F, I, P]
        lib.fa_forward_varlen.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, P]
        lib.fa_paged_prefill.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, I, P]
        lib.fa_paged_decode_workspace_size.argtypes = [I, I, I, I]
        lib.fa_paged_decode_workspace_size.restype = Z
        lib.fa_paged_decode.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, Z, P]
        lib.fa_paged_decode_fused.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, Z, P]
        lib.fa_paged_decode_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P]
        lib.fa_paged_gather.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, P]
        lib.fa_split_combine.argtypes = [P, P, P, P, P, I, I, I, I, P]
        lib.fa_last_error.argtypes = []
        lib.fa_last_error.restype = ctypes.c_char_p
        lib.fa_get_device_status.argtypes = [P, ctypes.POINTER(I)]
        for name in ("fa_forward", "fa_forward_fp8", "fa_forward_f32", "fa_forward_varlen",
                     "fa_paged_prefill",
                     "fa_paged_decode", "fa_paged_decode_fused",
                     "fa_paged_decode_noalloc", "fa_paged_gather", "fa_split_combine",
                     "fa_get_device_status"):
            getattr(lib, name).restype = I
        _lib = lib
        return lib


def _p(x):
    """Pointer of a tensor / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int):
    if rc != FA_OK:
        msg = load().fa_last_error()
        raise FaError(rc, msg.decode() if msg else "")


# ------------------------------------------------------------ C entry points
def fa_forward(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, scale, causal, stream=None):
    _check(load().fa_forward(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, Hkv, n, m, d, dv,
                             float(scale), int(causal), _stream(stream)))


def fa_forward_fp8(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, scale, q_descale, k_descale,
                   v_descale, causal, stream=None):
    _check(load().fa_forward_fp8(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, Hkv, n, m, d, dv,
                                 float(scale), float(q_descale), float(k_descale),
                                 float(v_descale), int(causal), _stream(stream)))


def fa_forward_f32(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, scale, causal, stream=None):
    _check(load().fa_forward_f32(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, Hkv, n, m, d, dv,
                                 float(scale), int(causal), _stream(stream)))


def fa_forward_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                      max_seqlen_q, max_seqlen_k, H, Hkv, d, dv, scale, causal, stream=None):
    _check(load().fa_forward_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu_seqlens_q),
                                    _p(cu_seqlens_k), num_seqs, total_q, total_k, max_seqlen_q,
                                    max_seqlen_k, H, Hkv, d, dv, float(scale), int(causal),
                                    _stream(stream)))


def fa_paged_prefill(q, k_cache, v_cache, block_table, seq_lens, cu_seqlens_q, o, lse, num_seqs,
                     total_q, max_seqlen_q, H, Hkv, d, dv, page_size, num_pages,
                     max_blocks_per_seq, scale, causal, stream=None):
    _check(load().fa_paged_prefill(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(seq_lens),
                                   _p(cu_seqlens_q), _p(o), _p(lse), num_seqs, total_q,
                                   max_seqlen_q, H, Hkv, d, dv, page_size, num_pages,
                                   max_blocks_per_seq, float(scale), int(causal), _stream(stream)))


def fa_paged_decode_workspace_size(num_seqs, H, dv, num_splits) -> int:
    return int(load().fa_paged_decode_workspace_size(num_seqs, H, dv, num_splits))


def fa_paged_decode(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, H, Hkv, d, dv,
                    page_size, num_pages, max_blocks_per_seq, num_splits, scale, workspace,
                    workspace_bytes, stream=None):
    _check(load().fa_paged_decode(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(seq_lens),
                                  _p(o), _p(lse), num_seqs, H, Hkv, d, dv, page_size, num_pages,
                                  max_blocks_per_seq, num_splits, float(scale), _p(workspace),
                                  int(workspace_bytes), _stream(stream)))


def fa_paged_decode_fused(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, H, Hkv, d,
                          dv, page_size, num_pages, max_blocks_per_seq, num_splits, scale,
                          workspace, workspace_bytes, stream=None):
    _check(load().fa_paged_decode_fused(_p(q), _p(k_cache), _p(v_cache), _p(block_table),
                                        _p(seq_lens), _p(o), _p(lse), num_seqs, H, Hkv, d, dv,
                                        page_size, num_pages, max_blocks_per_seq, num_splits,
                                        float(scale), _p(workspace), int(workspace_bytes),
                                        _stream(stream)))


def fa_paged_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, H, Hkv,
                            d, dv, page_size, num_pages, max_blocks_per_seq, num_splits, scale,
                            stream=None):
    """fa_paged_decode without a workspace: for callers that may not allocate
    device memory themselves.  The split partials live in the library's own
    fixed device array (FA_NOALLOC_SCRATCH_BYTES); calls share it, so calls
    that overlap on the GPU must not be issued."""
    _check(load().fa_paged_decode_noalloc(_p(q), _p(k_cache), _p(v_cache), _p(block_table),
                                          _p(seq_lens), _p(o), _p(lse), num_seqs, H, Hkv, d, dv,
                                          page_size, num_pages, max_blocks_per_seq, num_splits,
                                          float(scale), _stream(stream)))


def fa_paged_gather(k_cache, v_cache, block_table, seq_lens, k_out, v_out, num_seqs, Hkv, d,
                    page_size, num_pages, max_blocks_per_seq, num_splits, stream=None):
    _check(load().fa_paged_gather(_p(k_cache), _p(v_cache), _p(block_table), _p(seq_lens),
                                  _p(k_out), _p(v_out), num_seqs, Hkv, d, page_size, num_pages,
                                  max_blocks_per_seq, num_splits, _stream(stream)))


def fa_split_combine(part_m, part_l, part_o, o, lse, num_seqs, H, num_splits, dv, stream=None):
    _check(load().fa_split_combine(_p(part_m), _p(part_l), _p(part_o), _p(o), _p(lse), num_seqs, H,
                                   num_splits, dv, _stream(stream)))


def fa_get_device_status(stream=None) -> int:
    st = ctypes.c_int(0)
    _check(load().fa_get_device_status(_stream(stream), ctypes.byref(st)))
    return st.value


def fa_last_error() -> str:
    msg = load().fa_last_error()
    return msg.decode() if msg else ""


# ------------------------------------------------ torch-allocating helpers
def forward(q, k, v, scale, causal=False, stream=None):
    """q [B,n,H,d], k [B,m,Hkv,d], v [B,m,Hkv,dv] bf16 CUDA tensors -> (o bf16, lse fp32 [B,H,n])."""
    import torch
    B, n, H, d = q.shape
    _, m, Hkv, dv = v.shape
    o = torch.empty((B, n, H, dv), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
    fa_forward(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, scale, causal, stream)
    return o, lse


def forward_fp8(q, k, v, scale, q_descale, k_descale, v_descale, causal=False, stream=None):
    """e4m3 q [B,n,H,d], k/v [B,m,Hkv,d] (uint8 or float8 tensors) -> (o bf16, lse fp32)."""
    import torch
    B, n, H, d = q.shape
    _, m, Hkv, dv = v.shape
    o = torch.empty((B, n, H, dv), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
    fa_forward_fp8(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, scale, q_descale, k_descale, v_descale,
                   causal, stream)
    return o, lse


def forward_f32(q, k, v, scale, causal=False, stream=None):
    import torch
    B, n, H, d = q.shape
    _, m, Hkv, dv = v.shape
    o = torch.empty((B, n, H, dv), dtype=torch.float32, device=q.device)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
    fa_forward_f32(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, scale, causal, stream)
    return o, lse


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale,
                   causal=True, stream=None):
    """Packed q [Tq,H,d], k/v [Tk,Hkv,d] -> (o [Tq,H,dv] bf16, lse [H,Tq] fp32)."""
    import torch
    Tq, H, d = q.shape
    Tk, Hkv, dv = v.shape
    S = cu_seqlens_q.shape[0] - 1
    o = torch.empty((Tq, H, dv), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((H, Tq), dtype=torch.float32, device=q.device)
    fa_forward_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, S, Tq, Tk, max_seqlen_q,
                      max_seqlen_k, H, Hkv, d, dv, scale, causal, stream)
    return o, lse


def paged_prefill(q, k_cache, v_cache, block_table, seq_lens, cu_seqlens_q, max_seqlen_q, scale,
                  causal=True, stream=None):
    """q [Tq,H,d] packed by cu_seqlens_q; caches [P,Hkv,page,d] -> (o [Tq,H,dv], lse [H,Tq])."""
    import torch
    Tq, H, d = q.shape
    P, Hkv, page, dv = v_cache.shape
    S = cu_seqlens_q.shape[0] - 1
    o = torch.empty((Tq, H, dv), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((H, Tq), dtype=torch.float32, device=q.device)
    fa_paged_prefill(q, k_cache, v_cache, block_table, seq_lens, cu_seqlens_q, o, lse, S, Tq,
                     max_seqlen_q, H, Hkv, d, dv, page, P, block_table.shape[1], scale, causal,
                     stream)
    return o, lse


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, num_splits, scale, workspace=None,
                 stream=None):
    """q [S,H,d]; caches [P,Hkv,page,d]; block_table [S,max_blocks] int32; seq_lens [S] int32."""
    import torch
    S, H, d = q.shape
    P, Hkv, page, dv = v_cache.shape
    need = fa_paged_decode_workspace_size(S, H, dv, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    o = torch.empty((S, H, dv), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((S, H), dtype=torch.float32, device=q.device)
    fa_paged_decode(q, k_cache, v_cache, block_table, seq_lens, o, lse, S, H, Hkv, d, dv, page, P,
                    block_table.shape[1], num_splits, scale, workspace, workspace.numel(), stream)
    return o, lse


def paged_decode_fused(q, k_cache, v_cache, block_table, seq_lens, num_splits, scale,
                       workspace=None, stream=None):
    """As paged_decode, in one launch; a workspace passed in must have had its
    ticket words zeroed once (a new one is zeroed here)."""
    import torch
    S, H, d = q.shape
    P, Hkv, page, dv = v_cache.shape
    need = fa_paged_decode_workspace_size(S, H, dv, num_splits)
    if workspace is None:
        workspace = torch.zeros(max(need, 1), dtype=torch.uint8, device=q.device)
    o = torch.empty((S, H, dv), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((S, H), dtype=torch.float32, device=q.device)
    fa_paged_decode_fused(q, k_cache, v_cache, block_table, seq_lens, o, lse, S, H, Hkv, d, dv,
                          page, P, block_table.shape[1], num_splits, scale, workspace,
                          workspace.numel(), stream)
    return o, lse


def split_combine(part_m, part_l, part_o, stream=None):
    import torch
    S, H, X, dv = part_o.shape
    o = torch.empty((S, H, dv), dtype=torch.bfloat16, device=part_o.device)
    lse = torch.empty((S, H), dtype=torch.float32, device=part_o.device)
    fa_split_combine(part_m, part_l, part_o, o, lse, S, H, X, dv, stream)
    return o, lse


def decode_workspace_views(workspace, num_seqs, H, dv, num_splits):
    """Views (part_m, part_l, part_o) of a decode workspace, for inspection."""
    import torch

    def r256(x):
        return (x + 255) // 256 * 256
    tri = num_seqs * H * num_splits
    ws = workspace.view(torch.uint8)[r256(num_seqs * H * 4):]   # past the ticket words
    a = r256(tri * 4)
    pm = ws[:tri * 4].view(torch.float32).view(num_seqs, H, num_splits)
    pl = ws[a:a + tri * 4].view(torch.float32).view(num_seqs, H, num_splits)
    po = ws[2 * a:2 * a + tri * dv * 4].view(torch.float32).view(num_seqs, H, num_splits, dv)
    return pm, pl, po

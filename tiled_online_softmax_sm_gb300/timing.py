"""Device timing of every workload of the hot path, one table.

  python -m tiled_online_softmax_sm_gb300.timing [--iters 20] [--warmup 5]
  python -m tiled_online_softmax_sm_gb300.timing --naive [--iters 20] [--warmup 5]

Each workload runs on resident inputs from the seeded generators (the same
as the tests and the bench).  A row reports the median of `iters` timed
launches after `warmup` untimed ones.  The launches are queued back to back
on the current stream with a CUDA event between each pair, so every interval
is one launch's device time and not the host's call.  The fp32 workload is
tiny (its device time is below the host's call time) and is timed as graph
replays of 20 launches, per launch.  Inputs smaller than L2 (the n=m=2048
shapes, the fp32 case) stay L2-resident across launches; the long-context,
decode, prefill and ragged inputs are larger than L2.  Rates use nominal work:
4*n*m*d*H*B FLOPs (halved when causal; the ragged and paged rows sum their
sequences), and for the decode the K and V bytes of every valid token.
Nothing is checked here; parity lives in the tests.

--naive times instead the materialised-score path against fa_forward at N =
512, 2048 and 8192 (B=1, H=32, d=128, bf16, causal and not), the wall-clock
side of "S12 FlashAttention", 练习 3 and 它还解锁了什么 (the 2-4x said to come
from the HBM round trips of S): plain torch ops on the same inputs, S = (Q *
scale) K^T in bf16, the causal mask written into S in place, a softmax over
S (bf16 out, fp32 inside), then P V.  Each path gets its own best layout
(head-major copies for the torch matmuls, made outside the timed region).
"""
from __future__ import annotations

import argparse
import sys

import numpy as np
import torch

from . import binding as fb
from . import inputs as I


def _dev(t):
    if t.dtype == "bf16":
        return torch.from_numpy(t.data.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(t.data).cuda()


def _median_ms(fn, iters, warmup):
    # Launches are queued back to back with an event between each pair, so
    # the device never waits for the host's call and each interval is one
    # launch's device time; the warm-up launches are queued ahead of them.
    for _ in range(warmup):
        fn()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    evs[0].record()
    for i in range(iters):
        fn()
        evs[i + 1].record()
    torch.cuda.synchronize()
    return float(np.median([evs[i].elapsed_time(evs[i + 1]) for i in range(iters)]))


def _graph_median_ms(fn, iters, warmup, per_graph=20):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            fn()
    return _median_ms(g.replay, iters, 3) / per_graph


def _dense(c, iters, warmup):
    q, k, v = _dev(c.q), _dev(c.k), _dev(c.v)
    o = torch.empty((c.B, c.n, c.H, c.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((c.B, c.H, c.n), dtype=torch.float32, device="cuda")
    ms = _median_ms(lambda: fb.fa_forward(q, k, v, o, lse, c.B, c.H, c.Hkv, c.n, c.m, c.d, c.dv,
                                          c.scale, int(c.causal)), iters, warmup)
    flops = 4.0 * c.n * c.m * c.d * c.H * c.B / (2 if c.causal else 1)
    return ms, flops / (ms * 1e9), "TFLOP/s"


def rows(iters: int, warmup: int):
    out = []
    c = I.c1_fp32()
    q, k, v = _dev(c.q), _dev(c.k), _dev(c.v)
    o = torch.empty((c.B, c.n, c.H, c.dv), dtype=torch.float32, device="cuda")
    lse = torch.empty((c.B, c.H, c.n), dtype=torch.float32, device="cuda")
    ms = _graph_median_ms(lambda: fb.fa_forward_f32(q, k, v, o, lse, c.B, c.H, c.Hkv, c.n, c.m,
                                                    c.d, c.dv, c.scale, 0), iters, warmup)
    out.append(("fp32 n=m=256 d=64 (graph replay)", ms, 4.0 * c.n * c.m * c.d / (ms * 1e9), "TFLOP/s"))
    for causal in (False, True):
        out.append((f"bf16 B=4 H=16 n=m=2048 d=128 causal={causal}",) + _dense(I.c2_bf16(causal=causal), iters, warmup))
    out.append(("bf16 B=1 H=32 n=m=8192 d=128 causal",) + _dense(I.c3_bf16(), iters, warmup))
    # e4m3 forward, same long-context shape
    g = I.rng(I.BASE_SEED, 3)
    ts = [I.Tensor.from_f32(I.normal_f32(g, (1, 8192, 32, 128)), "e4m3") for _ in range(3)]
    q8, k8, v8 = (torch.from_numpy(t.data).cuda() for t in ts)
    o8 = torch.empty((1, 8192, 32, 128), dtype=torch.bfloat16, device="cuda")
    l8 = torch.empty((1, 32, 8192), dtype=torch.float32, device="cuda")
    ms = _median_ms(lambda: fb.fa_forward_fp8(q8, k8, v8, o8, l8, 1, 32, 32, 8192, 8192, 128, 128,
                                              I.fp32_scale(128), ts[0].descale, ts[1].descale,
                                              ts[2].descale, 1), iters, warmup)
    out.append(("e4m3 B=1 H=32 n=m=8192 d=128 causal", ms, 4.0 * 8192 * 8192 * 128 * 32 / 2 / (ms * 1e9), "TFLOP/s"))
    del q8, k8, v8, o8, l8
    # paged grouped-head decode at 4, 8, 16 splits
    dc = I.c4_decode(poison=False)
    qd, kc, vc = _dev(dc.q), _dev(dc.k_cache), _dev(dc.v_cache)
    bt = torch.from_numpy(dc.block_table).cuda()
    sl = torch.from_numpy(dc.seq_lens).cuda()
    S = len(dc.seq_lens)
    for X in (4, 8, 16):
        need = fb.fa_paged_decode_workspace_size(S, dc.H, dc.dv, X)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        od = torch.empty((S, dc.H, dc.dv), dtype=torch.bfloat16, device="cuda")
        ld = torch.empty((S, dc.H), dtype=torch.float32, device="cuda")
        ms = _median_ms(lambda: fb.fa_paged_decode(qd, kc, vc, bt, sl, od, ld, S, dc.H, dc.Hkv, dc.d,
                                                   dc.dv, dc.page_size, dc.num_pages, dc.max_blocks,
                                                   X, dc.scale, ws, need), iters, warmup)
        out.append((f"paged decode 64 seqs H=32 Hkv=8 splits={X}", ms, dc.kv_bytes / (ms * 1e6), "GB/s"))
    # the same decode in one launch (fa_paged_decode_fused), one zeroed workspace for all
    wsf = torch.zeros(fb.fa_paged_decode_workspace_size(S, dc.H, dc.dv, 16), dtype=torch.uint8,
                      device="cuda")
    for X in (4, 8, 16):
        od = torch.empty((S, dc.H, dc.dv), dtype=torch.bfloat16, device="cuda")
        ld = torch.empty((S, dc.H), dtype=torch.float32, device="cuda")
        ms = _median_ms(lambda: fb.fa_paged_decode_fused(qd, kc, vc, bt, sl, od, ld, S, dc.H, dc.Hkv,
                                                         dc.d, dc.dv, dc.page_size, dc.num_pages,
                                                         dc.max_blocks, X, dc.scale, wsf,
                                                         wsf.numel()), iters, warmup)
        out.append((f"paged decode fused 64 seqs H=32 Hkv=8 splits={X}", ms, dc.kv_bytes / (ms * 1e6), "GB/s"))
    # paged prefill: 512-token chunks of 16 sequences of the decode pool
    lens = I.uniform_lengths(63, 16, 512, 8192)
    ql = np.minimum(lens, 512)
    kv = I.decode_case(63, num_seqs=16, H=32, Hkv=8, d=128, lens=lens, max_blocks=512, poison=False)
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(cu[-1])
    qp = _dev(I.Tensor.from_f32(I.normal_f32(I.rng(63, 51), (T, 32, 128)), "bf16"))
    kp, vp = _dev(kv.k_cache), _dev(kv.v_cache)
    btp = torch.from_numpy(kv.block_table).cuda()
    slp = torch.from_numpy(kv.seq_lens).cuda()
    cut = torch.from_numpy(cu).cuda()
    op = torch.empty((T, 32, 128), dtype=torch.bfloat16, device="cuda")
    lp = torch.empty((32, T), dtype=torch.float32, device="cuda")
    ms = _median_ms(lambda: fb.fa_paged_prefill(qp, kp, vp, btp, slp, cut, op, lp, 16, T, 512, 32, 8,
                                                128, 128, 16, kv.num_pages, 512, kv.scale, 1),
                    iters, warmup)
    fl = sum(4.0 * int(nq) * 128 * 32 * (int(L) - int(nq) / 2) for nq, L in zip(ql, lens))
    out.append(("paged prefill 16 x 512-token chunks H=32 Hkv=8", ms, fl / (ms * 1e9), "TFLOP/s"))
    # ragged causal varlen
    for d in (64, 128):
        vcase = I.c5_varlen(d)
        qv, kvv, vv = _dev(vcase.q), _dev(vcase.k), _dev(vcase.v)
        cuv = torch.from_numpy(vcase.cu_seqlens).cuda()
        Tv = int(vcase.cu_seqlens[-1])
        mx = int(vcase.lens.max())
        ov = torch.empty((Tv, vcase.H, vcase.dv), dtype=torch.bfloat16, device="cuda")
        lv = torch.empty((vcase.H, Tv), dtype=torch.float32, device="cuda")
        ms = _median_ms(lambda: fb.fa_forward_varlen(qv, kvv, vv, ov, lv, cuv, cuv, len(vcase.lens), Tv,
                                                     Tv, mx, mx, vcase.H, vcase.Hkv, d, d, vcase.scale,
                                                     1), iters, warmup)
        fl = sum(4.0 * int(L) * int(L) * d * vcase.H / 2 for L in vcase.lens)
        out.append((f"ragged causal varlen 16 seqs H=16 d={d}", ms, fl / (ms * 1e9), "TFLOP/s"))
    return out


def fp8_gemm_peak(n: int = 8192, reps: int = 10):
    """Dense e4m3 GEMM rate of the library GEMM (cuBLASLt through
    torch._scaled_mm, bf16 out), n x n x n, best of reps: the denominator for
    the e4m3 forward's fraction.  None if this torch build has no e4m3 GEMM
    for the device."""
    try:
        a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn).t()   # column-major operand
        one = torch.ones((), device="cuda")
        mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        best = min(_median_ms(mm, 1, 0) for _ in range(reps))
        del a, b
        return 2.0 * n ** 3 / (best * 1e9)
    except (RuntimeError, AttributeError, TypeError) as e:  # no e4m3 GEMM in this build
        return None


def naive_vs_tiled(iters: int, warmup: int, sizes=(512, 2048, 8192), H: int = 32, D: int = 128):
    """Rows (N, causal, naive ms, tiled ms, S bytes) for the materialised-score
    path and fa_forward on the same bf16 inputs."""
    out = []
    scale = I.fp32_scale(D)
    for N in sizes:
        g = torch.Generator(device="cuda").manual_seed(N)
        q = torch.randn(1, N, H, D, device="cuda", generator=g).bfloat16()
        k = torch.randn(1, N, H, D, device="cuda", generator=g).bfloat16()
        v = torch.randn(1, N, H, D, device="cuda", generator=g).bfloat16()
        o = torch.empty_like(q)
        lse = torch.empty(1, H, N, device="cuda")
        qh, kh, vh = (x[0].transpose(0, 1).contiguous() for x in (q, k, v))   # [H, N, D]
        masked = torch.ones(N, N, dtype=torch.bool, device="cuda").tril().logical_not_()
        for causal in (True, False):
            def naive():
                s = torch.matmul(qh * scale, kh.transpose(-1, -2))           # [H, N, N] bf16
                if causal:
                    s.masked_fill_(masked, float("-inf"))
                p = torch.softmax(s, dim=-1)
                return torch.matmul(p, vh)

            naive_ms = _median_ms(naive, iters, warmup)
            tiled_ms = _median_ms(lambda: fb.fa_forward(q, k, v, o, lse, 1, H, H, N, N, D, D, scale,
                                                         int(causal)), iters, warmup)
            out.append((N, causal, naive_ms, tiled_ms, H * N * N * 2))
        del q, k, v, o, lse, qh, kh, vh, masked
        torch.cuda.empty_cache()
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--naive", action="store_true",
                    help="time the materialised-score path against fa_forward instead")
    ap.add_argument("--fp8-peak", action="store_true",
                    help="print the dense e4m3 GEMM rate of the library GEMM and exit")
    a = ap.parse_args(argv)
    if a.fp8_peak:
        r = fp8_gemm_peak()
        print(f"e4m3 GEMM 8192^3 (cuBLASLt via torch._scaled_mm): "
              + ("unavailable" if r is None else f"{r:.1f} TFLOP/s"))
        return 0
    if a.naive:
        print("| N | causal | materialised S (torch) | fa_forward | ratio | bf16 S size |\n"
              "|---|---|---|---|---|---|")
        for N, causal, naive_ms, tiled_ms, s_bytes in naive_vs_tiled(a.iters, a.warmup):
            print(f"| {N} | {causal} | {naive_ms:.3f} ms | {tiled_ms:.3f} ms | "
                  f"{naive_ms / tiled_ms:.1f}x | {s_bytes / 2**20:.0f} MiB |", flush=True)
        return 0
    print(f"| workload | median time | rate |\n|---|---|---|")
    for name, ms, rate, unit in rows(a.iters, a.warmup):
        t = f"{ms * 1000:.1f} us" if ms < 1 else f"{ms:.3f} ms"
        print(f"| {name} | {t} | {rate:.1f} {unit} |", flush=True)
    st = fb.fa_get_device_status()
    if st != 0:
        print(f"device status {st}")
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())

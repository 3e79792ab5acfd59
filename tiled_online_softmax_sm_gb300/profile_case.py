"""Run a few launches of one named workload on resident inputs, for profilers.

  python -m tiled_online_softmax_sm_gb300.profile_case fwd_c3 [--reps 2]

Workloads (sizes as in the bench and the parity tests):
  fwd_c3     causal bf16 forward, B=1 H=32 n=m=8192 d=128 (192 MB of inputs)
  fwd_c2     non-causal bf16 forward, B=4 H=16 n=m=2048 d=128
  fwd_c2c    causal bf16 forward, B=4 H=16 n=m=2048 d=128
  varlen_c5  ragged causal bf16 varlen forward, 16 sequences, d=128
  varlen_c5_d64  the same at d=64
  decode_c4  paged grouped-head decode, 64 sequences, H=32 Hkv=8, 8 splits (1.3 GB KV)
  fp8_c3     causal e4m3 forward, B=1 H=32 n=m=8192 d=128
  prefill_c4 paged prefill: 512-token chunks of 16 sequences of the decode pool
  fwd_f32    fp32 forward, n=m=256 d=64
Inputs come from the same seeded generators; nothing is checked here.
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


def make(name: str, splits: int = 8):
    if name in ("fwd_c3", "fwd_c2", "fwd_c2c"):
        c = I.c3_bf16() if name == "fwd_c3" else I.c2_bf16(causal=name == "fwd_c2c")
        q, k, v = _dev(c.q), _dev(c.k), _dev(c.v)
        o = torch.empty((c.B, c.n, c.H, c.dv), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((c.B, c.H, c.n), dtype=torch.float32, device="cuda")
        return lambda: fb.fa_forward(q, k, v, o, lse, c.B, c.H, c.Hkv, c.n, c.m, c.d, c.dv,
                                     c.scale, int(c.causal))
    if name in ("varlen_c5", "varlen_c5_d64"):
        c = I.c5_varlen(64 if name.endswith("d64") else 128)
        q, k, v = _dev(c.q), _dev(c.k), _dev(c.v)
        cu = torch.from_numpy(c.cu_seqlens).cuda()
        T = int(c.cu_seqlens[-1])
        mx = int(c.lens.max())
        o = torch.empty((T, c.H, c.dv), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((c.H, T), dtype=torch.float32, device="cuda")
        return lambda: fb.fa_forward_varlen(q, k, v, o, lse, cu, cu, len(c.lens), T, T, mx, mx,
                                            c.H, c.Hkv, c.d, c.dv, c.scale, 1)
    if name == "decode_c4":
        c = I.c4_decode()
        q, kc, vc = _dev(c.q), _dev(c.k_cache), _dev(c.v_cache)
        bt = torch.from_numpy(c.block_table).cuda()
        sl = torch.from_numpy(c.seq_lens).cuda()
        S = len(c.seq_lens)
        need = fb.fa_paged_decode_workspace_size(S, c.H, c.dv, splits)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        o = torch.empty((S, c.H, c.dv), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((S, c.H), dtype=torch.float32, device="cuda")
        return lambda: fb.fa_paged_decode(q, kc, vc, bt, sl, o, lse, S, c.H, c.Hkv, c.d, c.dv,
                                          c.page_size, c.num_pages, c.max_blocks, splits, c.scale,
                                          ws, need)
    if name == "fp8_c3":
        g = I.rng(I.BASE_SEED, 3)
        ts = [I.Tensor.from_f32(I.normal_f32(g, (1, 8192, 32, 128)), "e4m3") for _ in range(3)]
        q, k, v = (torch.from_numpy(t.data).cuda() for t in ts)
        o = torch.empty((1, 8192, 32, 128), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((1, 32, 8192), dtype=torch.float32, device="cuda")
        sc = I.fp32_scale(128)
        return lambda: fb.fa_forward_fp8(q, k, v, o, lse, 1, 32, 32, 8192, 8192, 128, 128, sc,
                                         ts[0].descale, ts[1].descale, ts[2].descale, 1)
    if name == "prefill_c4":
        lens = I.uniform_lengths(63, 16, 512, 8192)
        ql = np.minimum(lens, 512)
        kv = I.decode_case(63, num_seqs=16, H=32, Hkv=8, d=128, lens=lens, max_blocks=512)
        cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        T = int(cu[-1])
        q = _dev(I.Tensor.from_f32(I.normal_f32(I.rng(63, 51), (T, 32, 128)), "bf16"))
        kc, vc = _dev(kv.k_cache), _dev(kv.v_cache)
        bt = torch.from_numpy(kv.block_table).cuda()
        sl = torch.from_numpy(kv.seq_lens).cuda()
        cut = torch.from_numpy(cu).cuda()
        o = torch.empty((T, 32, 128), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((32, T), dtype=torch.float32, device="cuda")
        return lambda: fb.fa_paged_prefill(q, kc, vc, bt, sl, cut, o, lse, 16, T, 512, 32, 8, 128,
                                           128, 16, kv.num_pages, 512, kv.scale, 1)
    if name == "fwd_f32":
        c = I.c1_fp32()
        q, k, v = _dev(c.q), _dev(c.k), _dev(c.v)
        o = torch.empty((c.B, c.n, c.H, c.dv), dtype=torch.float32, device="cuda")
        lse = torch.empty((c.B, c.H, c.n), dtype=torch.float32, device="cuda")
        return lambda: fb.fa_forward_f32(q, k, v, o, lse, c.B, c.H, c.Hkv, c.n, c.m, c.d, c.dv,
                                         c.scale, 0)
    raise SystemExit(f"unknown workload {name}")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("workload")
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--splits", type=int, default=8)
    a = ap.parse_args(argv)
    fn = make(a.workload, a.splits)
    for _ in range(a.reps):
        fn()
    torch.cuda.synchronize()
    st = fb.fa_get_device_status()
    print(f"{a.workload}: {a.reps} launches, device status {st}")
    return 0 if st == 0 else 1


if __name__ == "__main__":
    sys.exit(main())

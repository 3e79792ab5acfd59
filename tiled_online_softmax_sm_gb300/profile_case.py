"""Run a few launches of one named workload on resident inputs, for profilers.

  python -m tiled_online_softmax_sm_gb300.profile_case fwd_c3 [--reps 2]

Workloads (sizes as in the bench and the parity tests):
  fwd_c3     causal bf16 forward, B=1 H=32 n=m=8192 d=128 (192 MB of inputs)
  fwd_c2     non-causal bf16 forward, B=4 H=16 n=m=2048 d=128
  fwd_c2c    causal bf16 forward, B=4 H=16 n=m=2048 d=128
  varlen_c5  ragged causal bf16 varlen forward, 16 sequences, d=128
  decode_c4  paged grouped-head decode, 64 sequences, H=32 Hkv=8, 8 splits (1.3 GB KV)
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
    if name == "varlen_c5":
        c = I.c5_varlen(128)
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

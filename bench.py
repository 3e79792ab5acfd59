"""Benchmark of the tiled online-softmax attention hot path on GB300.

One step = one pass of the whole hot path on resident synthetic inputs:
  * the long-context causal bf16 forward (B=1, H=32, n=m=8192, d=dv=128)
    through fa_forward, and
  * one paged grouped-head decode step (64 sequences, H=32, Hkv=8, d=128,
    page 16, context lengths uniform on [512, 8192], 8 splits) through
    fa_paged_decode (split partials + merge).
value = forward TFLOP/s (4*n*m*d*H/2 FLOPs, causal halved) from CUDA events
around each forward launch; the decode GB/s (K and V bytes of every valid
token) is reported beside it.  Every input (192 MB forward, 1.3 GB KV cache)
is larger than the 129 MB L2, and the decode step streams the cache between
two forwards.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle on the host cores on a bounded
sample of the same workload (the only other code this file may run).
Under torchrun each rank runs the same per-GPU workload (weak scaling, no
collective on the data path); rank 0 prints the JSON line.  At N=1 the line
also carries "configs": every workload of the path timed on the GPU (median
of 20 launches, as tiled_online_softmax_sm_gb300.timing reports them) beside
the oracle's rate on a bounded sample of the same inputs (--no-configs skips
it).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s & % bf16 tensor peak; paged decode HBM GB/s & % peak"
FWD_SHAPE = dict(B=1, H=32, n=8192, m=8192, d=128, causal=True)
DECODE_SPLITS = 8
def workload_name(splits: int) -> str:
    return ("long-context causal prefill bf16 B=1 H=32 n=m=8192 d=dv=128 + paged GQA decode "
            f"bf16 64 seqs H=32 Hkv=8 d=128 page 16 ctx U[512,8192] split {splits}")
FWD_KERNEL_SRC = os.path.join(ROOT, "tiled_online_softmax_sm_gb300", "csrc", "fwd_bf16_sm103.cu")
DEC_KERNEL_SRC = os.path.join(ROOT, "tiled_online_softmax_sm_gb300", "csrc", "decode.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def fwd_flops(B, H, n, m, d, causal, **_):
    f = 4.0 * n * m * d * H * B
    return f / 2 if causal else f


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_units(total: int, rank: int, world: int) -> range:
    """Contiguous near-equal slice of `total` independent units for `rank`."""
    lo = total * rank // world
    hi = total * (rank + 1) // world
    return range(lo, hi)


def reduce_max(values, device=None):
    """Element-wise max over ranks of a list of floats (identity without a
    process group).  Used for the timed region: the slowest rank decides."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def src_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(kernel_key, src_path):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source; otherwise None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t.get(kernel_key)
        if e and e.get("src_sha256_16") == src_hash(src_path):
            return e["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    return None


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(p[1]) for _, p in inside if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in inside if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in inside:
            for nm, val in zip(names, p[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# --------------------------------------------------------------- CPU oracle
def _oracle_rows(case, count, offset=0):
    """`count` query rows (b, h, i) evenly spread over the whole forward."""
    B, H, n = case.B, case.H, case.n
    total = B * H * n
    idx = (np.linspace(0, total - 1, count).astype(np.int64) + offset) % total
    return np.stack([idx // (H * n), (idx // n) % H, idx % n], 1).astype(np.int32)


def _rows_flops(case, rows):
    vis = (rows[:, 2].astype(np.float64) + 1) if case.causal else np.full(len(rows), case.m, np.float64)
    return float(np.sum(vis) * 2 * (case.d + case.dv))


def cpu_oracle_forward_sample(case, target_s: float = 8.0, offset: int = 0, count: int | None = None):
    """Time the float64 oracle on a bounded, evenly spread sample of the
    forward's query rows; returns (TFLOP/s, seconds, rows, threads).  Without
    `count`, the sample grows by doubling until it takes about target_s."""
    import oracle
    if count is None:
        count = 512
        while True:
            rows = _oracle_rows(case, count, offset)
            t = time.perf_counter()
            oracle.attention_rows(case.q.values, case.k.values, case.v.values, case.scale,
                                  case.causal, rows)
            dt = time.perf_counter() - t
            if dt >= target_s / 2 or count >= case.B * case.H * case.n:
                break
            count = min(case.B * case.H * case.n, count * 2)
    else:
        rows = _oracle_rows(case, count, offset)
        t = time.perf_counter()
        oracle.attention_rows(case.q.values, case.k.values, case.v.values, case.scale, case.causal,
                              rows)
        dt = time.perf_counter() - t
    return _rows_flops(case, rows) / dt / 1e12, dt, count, oracle.num_threads()


def cpu_oracle_decode_sample(case, target_s: float = 4.0):
    """Time the oracle's paged decode on a sample of sequences; returns GB/s of
    K/V bytes of the valid tokens processed."""
    import oracle
    S = len(case.seq_lens)
    take = 1
    while True:
        sel = np.arange(0, S, max(1, S // take))[:take]
        t = time.perf_counter()
        oracle.paged_decode(case.q.values[sel], case.k_cache.values, case.v_cache.values,
                            case.block_table[sel], case.seq_lens[sel], case.scale)
        dt = time.perf_counter() - t
        if dt * 2 > target_s or take >= S:
            break
        take = min(S, take * 2)
    nbytes = int(case.seq_lens[sel].sum()) * case.Hkv * (case.d + case.dv) * 2
    return nbytes / dt / 1e9, dt, len(sel)


def cpu_oracle_varlen_sample(case, target_s: float = 2.0):
    """Time the oracle's packed ragged attention on whole sequences, taken in
    index order and doubling in number until a run takes about target_s;
    returns (TFLOP/s, seconds, sequences)."""
    import oracle
    S = len(case.lens)
    take = 1
    while True:
        L = case.lens[:take]
        T = int(np.sum(L))
        cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
        t = time.perf_counter()
        oracle.varlen(case.q.values[:T], case.k.values[:T], case.v.values[:T], cu, cu, case.scale,
                      True)
        dt = time.perf_counter() - t
        if dt * 2 > target_s or take >= S:
            break
        take = min(S, take * 2)
    d, dv, H = case.q.values.shape[2], case.v.values.shape[2], case.q.values.shape[1]
    flops = sum(2.0 * int(x) * (int(x) + 1) * (d + dv) * H / 2 for x in L)
    return flops / dt / 1e12, dt, take


def config_table(peaks):
    """Every workload of the path on the GPU (median of 20 launches each, as
    the timing tool reports them, with the fraction of the measured peak that
    bounds it) beside the float64 oracle timed on a bounded sample of the
    same inputs on the host cores."""
    import oracle
    from tiled_online_softmax_sm_gb300 import inputs as I
    from tiled_online_softmax_sm_gb300 import timing

    # e4m3: the library's own dense e4m3 GEMM rate measured here, else the
    # nominal ratio (4.5 vs 2.25 PFLOP/s) times the measured bf16 peak
    fp8_peak = timing.fp8_gemm_peak()
    fp8_note = ("measured e4m3 GEMM (cuBLASLt) %.1f TFLOP/s" % fp8_peak if fp8_peak
                else "2 x the measured bf16 peak (no e4m3 GEMM measured)")

    def frac(name, rate, unit):
        if name.startswith("fp32"):
            return None   # a few microseconds: bound by latency, not by a pipe
        if unit == "GB/s":
            return round(rate / peaks["hbm_gbs"], 4)
        if name.startswith("e4m3"):
            return round(rate / (fp8_peak or 2.0 * peaks["bf16_tflops"]), 4)
        return round(rate / peaks["bf16_tflops"], 4)

    table = {name: {"gpu": {"ms": round(ms, 4), "rate": round(rate, 2), "unit": unit,
                            "frac": frac(name, rate, unit)}}
             for name, ms, rate, unit in timing.rows(20, 5)}
    for name in table:
        if name.startswith("e4m3"):
            table[name]["gpu"]["peak"] = fp8_note
    c1 = I.c1_fp32()
    c1_flops = 4.0 * 256 * 256 * 64
    all_threads = oracle.num_threads()
    for threads in (all_threads, 1):   # the small fp32 case on all cores and on one
        prev = oracle.set_num_threads(threads)
        try:
            t = time.perf_counter()
            oracle.attention(c1.q.values, c1.k.values, c1.v.values, c1.scale, False)
            dt = time.perf_counter() - t
        finally:
            oracle.set_num_threads(prev)
        key = "oracle" if threads == all_threads else "oracle_1_core"
        table["fp32 n=m=256 d=64 (graph replay)"][key] = {
            "rate": round(c1_flops / dt / 1e12, 6), "unit": "TFLOP/s", "seconds": round(dt, 4),
            "threads": threads, "sample": "the whole problem"}
    for causal in (False, True):
        c2 = I.c2_bf16(causal=causal)
        tf, dt, rows, _ = cpu_oracle_forward_sample(c2, target_s=2.0)
        table[f"bf16 B=4 H=16 n=m=2048 d=128 causal={causal}"]["oracle"] = {
            "rate": round(tf, 6), "unit": "TFLOP/s", "seconds": round(dt, 3),
            "sample": f"{rows} of {4 * 16 * 2048} query rows, evenly spread"}
    for d in (64, 128):
        c5 = I.c5_varlen(d)
        tf, dt, seqs = cpu_oracle_varlen_sample(c5, target_s=2.0)
        table[f"ragged causal varlen 16 seqs H=16 d={d}"]["oracle"] = {
            "rate": round(tf, 6), "unit": "TFLOP/s", "seconds": round(dt, 3),
            "sample": f"the first {seqs} of 16 sequences, all rows"}
    return table


# --------------------------------------------------------------- main arms
def build_inputs(rank: int, world: int = 1, seed: int | None = None):
    """This rank's share of the global job: the job is `world` independent
    copies of the per-GPU workload (forward batch + decode batch), each with
    its own seed (seed + copy); rank r takes copy r (weak scaling)."""
    from tiled_online_softmax_sm_gb300 import inputs as I
    (copy,) = shard_units(world, rank, world)
    seed = I.BASE_SEED if seed is None else seed
    fwd = I.dense_case(seed + copy, FWD_SHAPE["B"], FWD_SHAPE["H"], FWD_SHAPE["n"],
                       FWD_SHAPE["m"], FWD_SHAPE["d"], dtype="bf16", causal=True, stream=3,
                       name="c3")
    dec = I.c4_decode(seed=seed + copy)
    return fwd, dec


def run_reference(args, world, rank):
    """The float64 CPU oracle, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return 0
    fwd, dec = build_inputs(0, 1, args.seed)
    # one sample size for every step: the whole run stays within a few minutes
    per_step_s = min(8.0, max(0.05, 150.0 / max(1, args.steps + args.warmup)))
    _, _, count, threads = cpu_oracle_forward_sample(fwd, target_s=per_step_s)
    steps = []
    for s in range(args.warmup + args.steps):
        tf, dt, rows, threads = cpu_oracle_forward_sample(fwd, offset=7 * s, count=count)
        if s >= args.warmup:
            steps.append((tf, dt, rows))
    tf = statistics.median(x[0] for x in steps)
    gbs, ddt, seqs = cpu_oracle_decode_sample(dec, target_s=min(4.0, per_step_s))
    sample = (f"forward: {steps[0][2]} of {FWD_SHAPE['B'] * FWD_SHAPE['H'] * FWD_SHAPE['n']} query "
              f"rows per step, evenly spread; decode: {seqs} of 64 sequences")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tf, 6), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * statistics.median(x[1] for x in steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(args.splits), "l2": "n/a (CPU)"},
        "decode": {"value": round(gbs, 4), "unit": "GB/s"},
        "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import torch
    from tiled_online_softmax_sm_gb300 import binding as fb

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    fb.load()

    fwd, dec = build_inputs(rank, world, args.seed)

    def to_dev(t):
        return torch.from_numpy(t.data.view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = to_dev(fwd.q), to_dev(fwd.k), to_dev(fwd.v)
    B, H, n, m, d = fwd.B, fwd.H, fwd.n, fwd.m, fwd.d
    o = torch.empty((B, n, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=dev)
    dq, dkc, dvc = to_dev(dec.q), to_dev(dec.k_cache), to_dev(dec.v_cache)
    dbt = torch.from_numpy(dec.block_table).to(dev)
    dsl = torch.from_numpy(dec.seq_lens).to(dev)
    S = len(dec.seq_lens)
    ws_bytes = fb.fa_paged_decode_workspace_size(S, dec.H, dec.dv, args.splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    dout = torch.empty((S, dec.H, dec.dv), dtype=torch.bfloat16, device=dev)
    dlse = torch.empty((S, dec.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def forward():
        fb.fa_forward(q, k, v, o, lse, B, H, H, n, m, d, d, fwd.scale, 1, stream)

    def decode():
        fb.fa_paged_decode(dq, dkc, dvc, dbt, dsl, dout, dlse, S, dec.H, dec.Hkv, dec.d, dec.dv,
                           dec.page_size, dec.num_pages, dec.max_blocks, args.splits, dec.scale,
                           ws, ws_bytes, stream)

    warmup = max(3, args.warmup)
    for _ in range(warmup):
        forward()
        decode()
    torch.cuda.synchronize(dev)
    if fb.fa_get_device_status(stream) != 0:
        raise RuntimeError("device status set during warm-up")

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_id = vis.split(",")[local].strip() if vis else str(local)
    sampler = ClockSampler(smi_id)
    if rank == 0:
        sampler.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_start.record(stream)
    for s in range(K):
        a, b_, c = ev[s]
        a.record(stream)
        forward()
        b_.record(stream)
        decode()
        c.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    wall1 = time.time()
    if rank == 0:
        sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(K)]
    dec_ms = [ev[s][1].elapsed_time(ev[s][2]) for s in range(K)]
    status = fb.fa_get_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} during the timed region")

    # max over ranks of the timed region and of each part
    total_ms, fwd_sum, dec_sum = reduce_max([total_ms, sum(fwd_ms), sum(dec_ms)], device=dev)

    flops = fwd_flops(**FWD_SHAPE)
    fwd_tflops = flops * K * world / (fwd_sum / 1e3) / 1e12
    dec_gbs = dec.kv_bytes * K * world / (dec_sum / 1e3) / 1e9

    # ---- end to end through the C ABI with host buffers (pinned), forward.
    # Every step copies its Q, K, V in from pinned host memory, runs the
    # forward and copies O and LSE back out.  Steps are pipelined the way a
    # serving loop would run them: copies in on one stream, the kernel on a
    # second, copies out on a third, with two device buffer sets, so step
    # k+1's inputs cross the link while step k computes and drains.  Copy
    # engines on this part move ~210 GB/s host to device and ~190 back.
    e2e = None
    if rank == 0 or world > 1:
        hq = torch.from_numpy(fwd.q.data.view(np.int16)).pin_memory()
        hk = torch.from_numpy(fwd.k.data.view(np.int16)).pin_memory()
        hv = torch.from_numpy(fwd.v.data.view(np.int16)).pin_memory()
        ho = torch.empty(o.shape, dtype=torch.int16).pin_memory()
        hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        bufs = []
        for _ in range(2):
            qi, ki, vi = (torch.empty(x.shape, dtype=torch.int16, device=dev) for x in (hq, hk, hv))
            bufs.append((qi, ki, vi, torch.empty_like(o), torch.empty_like(lse)))
        s_in, s_fwd, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev = lambda: torch.cuda.Event()
        ev_in, ev_fwd, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        started = [False, False]

        def e2e_step(step):
            bi = step & 1
            qi, ki, vi, ob, lb = bufs[bi]
            if started[bi]:
                s_in.wait_event(ev_fwd[bi])    # the forward of step-2 has read these inputs
                s_fwd.wait_event(ev_out[bi])   # and its O, LSE have left the device
            started[bi] = True
            with torch.cuda.stream(s_in):
                qi.copy_(hq, non_blocking=True)
                ki.copy_(hk, non_blocking=True)
                vi.copy_(hv, non_blocking=True)
                ev_in[bi].record(s_in)
            s_fwd.wait_event(ev_in[bi])
            fb.fa_forward(qi, ki, vi, ob, lb, B, H, H, n, m, d, d, fwd.scale, 1, s_fwd)
            ev_fwd[bi].record(s_fwd)
            s_out.wait_event(ev_fwd[bi])
            with torch.cuda.stream(s_out):
                ho.copy_(ob.view(torch.int16), non_blocking=True)
                hl.copy_(lb, non_blocking=True)
                ev_out[bi].record(s_out)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        KE = max(1, min(K, 20))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        for x in (s_in, s_fwd, s_out):
            x.wait_stream(torch.cuda.current_stream(dev))
        e0.record(s_in)
        s_fwd.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(KE):
            e2e_step(i)
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_fwd)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        if fb.fa_get_device_status(s_fwd) != 0:
            raise SystemExit("device status set during the end-to-end leg")
        e2e_ms = e0.elapsed_time(e1) / KE
        h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2
        d2h = ho.numel() * 2 + hl.numel() * 4
        e2e = {"value": round(flops / (e2e_ms / 1e3) / 1e12 * world, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_ms, 4),
               "pipelined": "copies in, forward and copies out on three streams, two buffer sets"}

    # ---- end to end, decode: the step's new query tokens, block tables and
    # sequence lengths come from pinned host memory and its O and LSE go back
    # to it, every step, through fa_paged_decode; the KV cache stays resident
    # on the device, as a serving cache does.  The copies are small (~1.2 MB a
    # step) beside the 1.17 GB of K/V the step reads; they overlap the
    # neighbouring steps' decodes.
    e2e_decode = None
    if rank == 0 or world > 1:
        hdq = torch.from_numpy(dec.q.data.view(np.int16)).pin_memory()
        hbt = torch.from_numpy(dec.block_table).pin_memory()
        hsl = torch.from_numpy(dec.seq_lens).pin_memory()
        hdo = torch.empty(dout.shape, dtype=torch.int16).pin_memory()
        hdl = torch.empty(dlse.shape, dtype=torch.float32).pin_memory()
        # pipelined like the forward's leg: copies in on one stream, the
        # decodes (one after another, so they share the workspace) on a
        # second, copies out on a third, with two sets of step buffers
        dbufs = []
        for _ in range(2):
            dbufs.append((torch.empty_like(dq).view(torch.int16), torch.empty_like(dbt),
                          torch.empty_like(dsl), torch.empty_like(dout), torch.empty_like(dlse)))
        t_in, t_dec, t_out = (torch.cuda.Stream(dev) for _ in range(3))
        dev_in, dev_dec, dev_out = ([torch.cuda.Event(), torch.cuda.Event()] for _ in range(3))
        dstarted = [False, False]

        def e2e_decode_step(step):
            bi = step & 1
            qb, btb, slb, ob, lb = dbufs[bi]
            if dstarted[bi]:
                t_in.wait_event(dev_dec[bi])    # the decode of step-2 has read these inputs
                t_dec.wait_event(dev_out[bi])   # and its O, LSE have left the device
            dstarted[bi] = True
            with torch.cuda.stream(t_in):
                qb.copy_(hdq, non_blocking=True)
                btb.copy_(hbt, non_blocking=True)
                slb.copy_(hsl, non_blocking=True)
                dev_in[bi].record(t_in)
            t_dec.wait_event(dev_in[bi])
            fb.fa_paged_decode(qb.view(torch.bfloat16), dkc, dvc, btb, slb, ob, lb, S, dec.H,
                               dec.Hkv, dec.d, dec.dv, dec.page_size, dec.num_pages, dec.max_blocks,
                               args.splits, dec.scale, ws, ws_bytes, t_dec)
            dev_dec[bi].record(t_dec)
            t_out.wait_event(dev_dec[bi])
            with torch.cuda.stream(t_out):
                hdo.copy_(ob.view(torch.int16), non_blocking=True)
                hdl.copy_(lb, non_blocking=True)
                dev_out[bi].record(t_out)

        for x in (t_in, t_dec, t_out):
            x.wait_stream(torch.cuda.current_stream(dev))
        for i in range(3):
            e2e_decode_step(i)
        torch.cuda.synchronize(dev)
        KD = max(1, min(K, 50))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(t_in)
        t_dec.wait_event(e0)
        t_out.wait_event(e0)
        for i in range(KD):
            e2e_decode_step(i)
        t_out.wait_stream(t_in)
        t_out.wait_stream(t_dec)
        e1.record(t_out)
        torch.cuda.synchronize(dev)
        if fb.fa_get_device_status(t_dec) != 0:
            raise SystemExit("device status set during the end-to-end decode leg")
        ed_ms = e0.elapsed_time(e1) / KD
        h2d = hdq.numel() * 2 + hbt.numel() * 4 + hsl.numel() * 4
        d2h = hdo.numel() * 2 + hdl.numel() * 4
        e2e_decode = {"value": round(dec.kv_bytes * world / (ed_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                      "ms_per_step": round(ed_ms, 4),
                      "path": "q, block table, seq lens in and O, LSE out through pinned host "
                              "buffers each step; KV cache resident; copies pipelined across "
                              "steps on three streams, two buffer sets"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks = measured_peaks()
    fwd_avg = fwd_sum / K
    dec_avg = dec_sum / K
    achieved = flops / (fwd_avg / 1e3) / 1e12
    dec_achieved = dec.kv_bytes / (dec_avg / 1e3) / 1e9
    tr_fwd = traffic_for("fa_forward_c3", FWD_KERNEL_SRC)
    tr_dec = traffic_for("fa_paged_decode_c4", DEC_KERNEL_SRC)
    clocks = sampler.summary(wall0, wall1)

    # CPU baseline: the float64 oracle on a bounded sample of the forward
    tf_cpu, dt_cpu, rows_cpu, threads = cpu_oracle_forward_sample(fwd, target_s=8.0)

    # every workload of the path, GPU and oracle side by side (after the timed
    # region, one GPU only)
    configs = None
    if world == 1 and args.configs:
        # the table is extra evidence: a failure in it is reported in the line
        # rather than costing the line itself
        try:
            configs = config_table(peaks)
            gbs, ddt, seqs = cpu_oracle_decode_sample(dec, target_s=2.0)
            for name in configs:
                if name.startswith("paged decode"):
                    configs[name]["oracle"] = {"rate": round(gbs, 4), "unit": "GB/s",
                                               "seconds": round(ddt, 3),
                                               "sample": f"{seqs} of 64 sequences, unsplit"}
        except Exception as e:  # noqa: BLE001
            configs = {"error": f"{type(e).__name__}: {e}"}

    line = {
        "metric": METRIC,
        "value": round(fwd_tflops, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": warmup,
        "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(args.splits), "fwd_ms": round(fwd_avg, 4),
                   "decode_ms": round(dec_avg, 4), "decode_splits": args.splits,
                   "l2": "inputs larger than L2 (forward 192 MB, KV cache 1.3 GB streamed each step)"},
        "decode": {"value": round(dec_gbs, 2), "unit": "GB/s", "kv_bytes": int(dec.kv_bytes),
                   "frac_of_hbm_peak": round(dec_achieved / peaks["hbm_gbs"], 4)},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": tr_fwd, "kernel": "fwd_bf16_kernel<128, false, false, false>",
                     "peak_source": f"{peaks['source']} bf16 burst",
                     "flops_per_launch": flops},
        "roofline_decode": {"bound": "hbm", "achieved": round(dec_achieved, 2),
                            "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(dec_achieved / peaks["hbm_gbs"], 4), "traffic": tr_dec,
                            "kernel": "decode_partials_kernel + split_combine_kernel",
                            "peak_source": f"{peaks['source']} copy",
                            "bytes_per_launch": int(dec.kv_bytes)},
        "cpu_baseline": {"value": round(tf_cpu, 6), "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "cpu": cpu_model(),
                         "sample": f"{rows_cpu} evenly spread query rows of the forward "
                                   f"({dt_cpu:.1f} s)"},
        "e2e": e2e,
        "e2e_decode": e2e_decode,
        "gpu_launches": 3 * K,
        "clocks": clocks,
    }
    if configs is not None:
        line["configs"] = configs
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--splits", type=int, default=DECODE_SPLITS,
                    help="KV splits of the decode step (1..64)")
    ap.add_argument("--seed", type=int, default=None,
                    help="base seed of the synthetic inputs (default: the generators' own)")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the per-workload GPU and oracle table (N=1 only)")
    args = ap.parse_args(argv)
    if not 1 <= args.splits <= 64:
        ap.error(f"--splits {args.splits}: the decode takes 1..64 splits")
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    return args


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_info()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())

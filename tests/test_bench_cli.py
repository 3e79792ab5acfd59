"""Host logic of bench.py that needs no GPU: its command line, the workload
name each arm reports, and the rule that a traffic figure is reported only
for the kernel source it was captured on."""
import json

import pytest

import bench


def test_defaults_run_one_gpu_within_minutes():
    a = bench.parse_args([])
    assert (a.gpus, a.steps, a.warmup, a.impl) == (1, 1000, 10, "ours")
    assert (a.splits, a.seed, a.configs) == (bench.DECODE_SPLITS, None, True)
    assert a.warmup >= 3


def test_flags():
    a = bench.parse_args(["--impl", "reference", "--splits", "4", "--seed", "7", "--no-configs",
                          "--steps", "5", "--warmup", "3"])
    assert (a.impl, a.splits, a.seed, a.configs, a.steps, a.warmup) == \
        ("reference", 4, 7, False, 5, 3)


@pytest.mark.parametrize("argv", [["--splits", "0"], ["--splits", "65"], ["--steps", "0"],
                                  ["--warmup", "-1"], ["--impl", "other"]])
def test_bad_flags_are_refused(argv):
    with pytest.raises(SystemExit):
        bench.parse_args(argv)


def test_workload_name_names_the_split_count():
    assert bench.workload_name(8).endswith("split 8")
    assert bench.workload_name(16).endswith("split 16")
    assert "n=m=8192" in bench.workload_name(8) and "64 seqs" in bench.workload_name(8)


def test_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    table = tmp_path / "traffic.json"
    table.write_text(json.dumps({"k": {"src_sha256_16": bench.src_hash(str(src)),
                                       "dram_bytes_per_launch": 1234}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(table))
    assert bench.traffic_for("k", str(src)) == 1234
    assert bench.traffic_for("other", str(src)) is None
    src.write_text("// kernel v2\n")          # the kernel changed since the capture
    assert bench.traffic_for("k", str(src)) is None


def test_peaks_have_the_roofline_denominators():
    p = bench.measured_peaks()
    assert p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0 and p["source"] in ("measured", "fallback")


def test_forward_work_is_the_nominal_halved_count():
    """4 n m d H B FLOPs, halved when causal: 549.76 GFLOP for the causal
    B=1 H=32 n=m=8192 d=128 forward the bench times."""
    assert bench.fwd_flops(**bench.FWD_SHAPE) == 4.0 * 8192 * 8192 * 128 * 32 / 2 == 549755813888.0
    assert bench.fwd_flops(B=4, H=16, n=2048, m=2048, d=128, causal=False) == 137438953472.0

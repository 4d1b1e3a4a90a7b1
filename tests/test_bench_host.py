"""Host-side logic of the benchmark and the binding, on CPU.

* the algorithmic work model (FLOPs and bytes per stage) gives the path totals the
  hot-path scope fixes for the long-text workload, and the roofline is the slower of
  FLOPs at the bf16 peak and bytes at HBM bandwidth;
* a DRAM-traffic figure recorded from ncu is used only while the kernel's sources are
  unchanged;
* the whole-job value counts every rank's tokens over the slowest rank's time;
* the binding refuses to run without the native library (no fallback).
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from lsh_attention_04_b300 import inputs as gen  # noqa: E402


def test_work_model_long_text_totals():
    w = gen.WORKLOADS["long_B1_H8_L65536_d128_R8"]
    k = bench.work(w)
    N, R, d, nb, c = w.tokens, w.n_rounds, w.d, w.n_buckets, w.chunk
    # hash: N*R*(nb/2) dot products of length d; attention: QK^T and PV over c x 2c
    assert k["hash"]["flops"] == N * R * d * nb == 549_755_813_888
    assert k["attn"]["flops"] == 8 * N * R * c * d == 274_877_906_944
    total_f = sum(v["flops"] for v in k.values())
    assert total_f == 824_633_720_832                      # 825 GFLOP at this size
    total_b = sum(v["bytes"] for v in k.values())
    assert 2.9e9 < total_b < 3.0e9                         # ~2.95 GB: the o_r round trip dominates
    # roofline: slower of the two, with the measured peaks
    peaks, _ = bench.load_peaks()
    t_f = total_f / (peaks["bf16_tflops"] * 1e12)
    t_b = total_b / (peaks["hbm_gbs"] * 1e9)
    assert t_f > 0 and t_b > 0


def test_work_model_backward_totals():
    """Backward at the long-text shape: the hash and sort as in the forward pass, then five
    window contractions per token and round (20 c d flops) in the attention backward."""
    w = gen.WORKLOADS[gen.HEADLINE]
    wk = bench.work_backward(w)
    assert set(wk) == {"hash", "sort", "attn_bwd"}
    fwd = bench.work(w)
    assert wk["hash"] == fwd["hash"] and wk["sort"] == fwd["sort"]
    N = 8 * 65536
    assert wk["attn_bwd"]["flops"] == 20 * N * 8 * 64 * 128 == 687_194_767_360
    # qk, v bf16; out, g_out, dqk, dv fp32; lse, g_lse, inverse norms; buckets, perm
    assert wk["attn_bwd"]["bytes"] == N * (2 * 128 * 2 + 4 * 128 * 4 + 3 * 4 + 2 * 8 * 4)


def test_recorded_traffic_needs_unchanged_sources(tmp_path, monkeypatch):
    rec = {"wl": {"attn": {"bytes_per_launch": 123, "source_sha1": bench.source_digest("attn")}}}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("wl", "attn") == 123
    assert bench.recorded_traffic("wl", "hash") is None            # no record
    assert bench.recorded_traffic("other", "attn") is None
    monkeypatch.setattr(bench, "source_digest", lambda stage: "0" * 40)
    assert bench.recorded_traffic("wl", "attn") is None            # sources changed


def test_kernel_sources_exist():
    for stage, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "lsh_attention_04_b300", "csrc", f)), (stage, f)


def test_job_value_counts_all_ranks():
    assert bench.job_value(1000, 1, 2.0) == pytest.approx(500_000)
    assert bench.job_value(1000, 4, 2.0) == pytest.approx(2_000_000)


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    import lsh_attention_04_b300 as lsh
    monkeypatch.setattr(lsh, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(lsh, "_lib", None, raising=False)
    with pytest.raises(OSError):
        lsh.load()


def test_reference_arm_times_the_oracle_backward(capsys, monkeypatch):
    """--impl reference --pass backward on rank 0: the oracle's backward pass on a bounded
    sample, printed as one JSON line with the backward metric and a one-core baseline."""
    monkeypatch.setenv("RANK", "0")
    w = gen.Workload("tiny_bf16_B1_H1_L256_d64_R2", 1, 1, 256, 64, "bf16", 8, 2, 64, True, 4, 3)

    class A:
        gpus, steps, warmup, pass_ = 1, 1, 0, "backward"

    assert bench.run_reference(A, w) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC_BWD
    assert line["value"] > 0 and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert "backward" in line["cpu_baseline"]["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0

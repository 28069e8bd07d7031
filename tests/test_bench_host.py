"""Host logic of bench.py on CPU: the clock record's summary, the kernel
source hash that keys the stored DRAM counters, the counters' lookup, the
algorithmic byte counts of the timed kernels, and the reference arm's JSON
line (the CPU oracle timed on a row sample)."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _sampler_on(path):
    s = bench.ClockSampler(0, enabled=False)
    s.path = str(path)
    s.proc = object()  # a record exists; summary() only reads the file
    return s


def test_clock_summary_median_max_and_reasons(tmp_path):
    # index, clocks.sm, clocks.max.sm, power, active mask, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    rows = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active",  # unreadable: skipped
        "garbage line",
    ]
    p = tmp_path / "clocks.csv"
    p.write_text("\n".join(rows) + "\n")
    s = _sampler_on(p).summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_flags_slowdowns(tmp_path):
    p = tmp_path / "clocks.csv"
    p.write_text("0, 1500, 2070, 1000, 0x8, Active, Not Active, Active, Not Active\n"
                 "0, 1600, 2070, 1000, 0x8, Not Active, Active, Not Active, Not Active\n")
    s = _sampler_on(p).summary()
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1550.0 and s["samples"] == 2


def test_clock_summary_without_record(tmp_path):
    assert bench.ClockSampler(0, enabled=False).summary() is None
    p = tmp_path / "empty.csv"
    p.write_text("")
    assert _sampler_on(p).summary() is None


def _fake_tree(root, code):
    csrc = root / "row_wise_normalization_rmsnorm_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    (csrc / "k.cu").write_text(code)
    return root


def test_source_hash_ignores_comments_and_spacing(tmp_path, monkeypatch):
    base = "__global__ void k(float *y) {\n    y[0] = 1.f;  // one\n}\n"
    monkeypatch.setattr(bench, "ROOT", str(_fake_tree(tmp_path / "a", base)))
    h0 = bench.kernel_source_hash()
    reworded = "/* a kernel */\n__global__   void k(float *y) {\n\n    y[0] = 1.f;  // the value one\n}\n"
    monkeypatch.setattr(bench, "ROOT", str(_fake_tree(tmp_path / "b", reworded)))
    assert bench.kernel_source_hash() == h0
    changed = "__global__ void k(float *y) {\n    y[0] = 2.f;  // one\n}\n"
    monkeypatch.setattr(bench, "ROOT", str(_fake_tree(tmp_path / "c", changed)))
    assert bench.kernel_source_hash() != h0


def test_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    root = _fake_tree(tmp_path, "__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    (root / "profiles").mkdir()
    rec = {"source_hash": bench.kernel_source_hash(),
           "kernels": {"fwd": {"dram_bytes_per_launch": 476677120}}}
    (root / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("fwd") == 476677120
    assert bench.ncu_traffic("bwd") is None
    rec["source_hash"] = "0" * 16
    (root / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("fwd") is None
    (root / "profiles" / "dram_traffic.json").unlink()
    assert bench.ncu_traffic("fwd") is None


@pytest.mark.parametrize("M,N,s,P", [(16384, 8192, 2, 152), (7, 3, 4, 5), (1, 1, 2, 1)])
def test_algorithmic_bytes(M, N, s, P):
    # forward: x read, y written, w read, fp32 rstd written
    assert bench.bytes_fwd(M, N, s) == M * N * s + M * N * s + N * s + M * 4
    # backward main kernel: x and dy read, dx written, w and rstd read, P
    # fp32 partial rows written; the finalizer reads them and writes dW
    assert bench.bytes_bwd_main(M, N, s, P) == 3 * M * N * s + N * s + M * 4 + P * N * 4
    assert bench.bytes_bwd_finalize(N, s, P) == P * N * 4 + N * s
    assert bench.bytes_bwd(M, N, s, P) == bench.bytes_bwd_main(M, N, s, P) + bench.bytes_bwd_finalize(N, s, P)


def test_whole_job_throughput_scales_with_ranks():
    one = bench.whole_job_gbs(1_353_000_000, 1, 0.2097)
    assert abs(one - 1_353_000_000 / 0.2097e-3 / 1e9) < 1e-6
    assert abs(bench.whole_job_gbs(1_353_000_000, 4, 0.2097) - 4 * one) < 1e-6


def test_peak_falls_back_without_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6708.2}))
    assert bench.peaks() == (6708.2, "measured")


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the CPU oracle on a bounded row
    sample of the bench workload and prints one JSON line with the same
    metric and unit as the GPU arm, its own cpu_baseline and an e2e with no
    host-device copies; it needs no GPU."""
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3 and d["gpu_launches"] == 0
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["data"] == "synthetic"
    assert "16384x8192" in d["metric"] and d["config"]["M"] == 16384 and d["config"]["N"] == 8192
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}

"""Host-side pieces of the benchmark that need no GPU: the algorithmic work the
roofline divides by, the traffic lookup from the committed ncu summary (and
its refusal once the kernel source has changed), and the peak fallback."""
import hashlib
import json
import os

import numpy as np
import pytest

import bench
from vision_encoder_varlen_gb300 import workloads as wl


def test_algorithmic_flops_split_by_kernel():
    w = wl.make_config(5)
    L = w.lengths.astype(np.float64)
    total = bench.kernel_algorithmic_flops(w, "attn_long", 0)
    assert total == pytest.approx(w.useful_flops)                 # split 0: every segment is long
    assert total == pytest.approx(4 * np.sum(L * L) * 16 * 80)
    long64 = bench.kernel_algorithmic_flops(w, "attn_long", 64)
    short64 = bench.kernel_algorithmic_flops(w, "attn_tiny", 64)
    assert long64 + short64 == pytest.approx(total)
    w7 = wl.make_config(7)
    assert bench.kernel_algorithmic_flops(w7, "attn_long", 64) == 0.0     # all of it is tiny


def test_traffic_lookup_follows_the_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// one version\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    entry = {"workload": "w", "bytes_per_launch": 123.0, "source": "kernel.cu", "source_sha256_16": h}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"attn_long": [entry]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("attn_long", "w") == 123.0
    assert bench.load_traffic("attn_long", "other") is None
    assert bench.load_traffic("attn_tiny", "w") is None
    src.write_text("// another version\n")                        # the kernel changed since the capture
    assert bench.load_traffic("attn_long", "w") is None


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for kernel, entries in d.items():
        for e in entries:
            assert os.path.exists(os.path.join(bench.ROOT, e["source"])), e
            assert e["bytes_per_launch"] > 0


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert peaks["hbm_gbs"] > 0 and peaks["bf16_tflops_sustained"] > 0
    assert "fallback" in src


def test_clock_sampler_summary_and_missing_tool(tmp_path, monkeypatch):
    # the summary of a sampled CSV: median SM clock under load, the max, the active reasons
    s = bench.ClockSampler(0)
    path = tmp_path / "clocks.csv"
    rows = ["0, 2032, 2070, 1100.5, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2040, 2070, 1150.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 345, 2070, 90.0, 0x1, Not Active, Not Active, Not Active, Not Active",   # idle sample
            "0, 2010, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active",
            "garbage line"]
    path.write_text("\n".join(rows) + "\n")
    s.proc, s.path = object(), str(path)
    got = s.summary()
    assert got == {"sm_mhz": 2032.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 4}
    assert not path.exists()                               # the temporary file is removed
    # without nvidia-smi the sampler reports nothing and leaves no file behind
    monkeypatch.setattr(bench.subprocess, "Popen", lambda *a, **k: (_ for _ in ()).throw(FileNotFoundError()))
    with bench.ClockSampler(0) as c:
        pass
    assert c.summary() is None and c.path is None


def test_roofline_denominator_follows_the_timed_region():
    # a contraction timed for less than SUSTAINED_AFTER_S is held to the burst peak, a longer
    # timed region to the sustained one; both are named in the entry
    w = wl.make_config(3)
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    kt = {"attn_long": (10, 0.5), "qk_norm_rope": (10, 0.2)}
    short = bench.roofline_entry(None, w, kt, 64, peaks, "measured", 0.3, False)
    long_ = bench.roofline_entry(None, w, kt, 64, peaks, "measured", 2.5, False)
    assert short["kernel"] == "attn_long" and short["bound"] == "tensor"
    assert short["peak"] == 1900.0 and "bf16_tflops " in short["peak_source"]
    assert long_["peak"] == 1700.0 and "bf16_tflops_sustained" in long_["peak_source"]
    alg = bench.kernel_algorithmic_flops(w, "attn_long", 64)
    assert short["achieved"] == pytest.approx(alg / 0.05e-3 / 1e12)
    assert short["frac"] == pytest.approx(short["achieved"] / 1900.0)
    # an HBM-bound dominant kernel is held to the copy bandwidth
    hb = bench.roofline_entry(None, w, {"qk_norm_rope": (4, 0.4)}, 64, peaks, "measured", 0.1, False)
    assert hb["bound"] == "hbm" and hb["peak"] == 6800.0
    assert hb["achieved"] == pytest.approx(8.0 * w.total_tokens * 16 * 80 / 0.1e-3 / 1e9)


def test_both_arms_describe_the_same_workload():
    import argparse
    args = argparse.Namespace(interleaved=False, lse=False, fused_q=False)
    w = wl.make_config(5)
    a, b = bench.config_dict(w, args, 1), bench.config_dict(w, args, 1)
    assert a == b and a["workload"] == w.name and a["useful_flops_per_step"] == w.useful_flops
    assert "inputs larger than L2" in a["l2"]
    assert "flushed" in bench.config_dict(wl.make_config(2), args, 1)["l2"]

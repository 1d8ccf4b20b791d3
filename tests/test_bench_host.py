"""Host-side pieces of bench.py, on the CPU: the byte model of a cached row,
peak loading, the clock-log summary, the kernel-source hash that keys the
committed traffic counters, and the JSON line of the reference arm."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_row_bytes_and_visible_keys():
    # codes + bf16 scale and bias per 64-group, for K and for V
    assert bench.rb_pair(512, 4) == 576 and bench.rb_pair(512, 8) == 1088
    assert bench.rb_pair(256, 4) == 288 and bench.rb_pair(256, 8) == 544
    assert bench.visible_keys(0, 0) == 1 and bench.visible_keys(99, 0) == 100
    assert bench.visible_keys(99, 64) == 64 and bench.visible_keys(10, 64) == 11


def test_peaks_fallback_and_measured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == bench.FALLBACK_HBM_GBS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"gb300": {"hbm_gbs": 7100.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1750.0}}))
    p = bench.load_peaks()
    # the burst bf16 figure (kernels are timed inside sub-millisecond steps)
    assert p == {"hbm_gbs": 7100.0, "bf16_tflops": 2000.0, "source": "measured"}


def test_clock_summary():
    c = bench.ClockSampler(0)
    c.lines = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 2040, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_code_only_ignores_comments_and_layout():
    a = 'int a = 1; // note\n/* block\n comment */ const char* s = "/* kept */ // kept";\n'
    b = 'int  a = 1;\nconst char* s = "/* kept */ // kept";'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(a.replace("a = 1", "a = 2"))
    assert "/* kept */ // kept" in bench._code_only(a)


def test_traffic_only_for_the_kernel_sources_it_was_taken_on(tmp_path, monkeypatch):
    h = bench.source_hash("decode_kernel_512")
    assert h is not None and bench.source_hash("no_such_kernel") is None
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for key, e in t.get("decode_kernel_512", {}).items():
        got = bench.traffic_for("decode_kernel_512", key, 1e9)
        if e["source_hash"] == h:
            assert got == pytest.approx(e["traffic_over_algorithmic"] * 1e9)
        else:
            assert got is None
    # a planted entry: used on the current sources only, keyed by bit width
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"decode_kernel_512": {
        "8bit": {"source_hash": h, "traffic_over_algorithmic": 1.01},
        "4bit": {"source_hash": "0" * 16, "traffic_over_algorithmic": 1.02}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda k: h if k == "decode_kernel_512" else None)
    assert bench.traffic_for("decode_kernel_512", "8bit", 2e9) == pytest.approx(2.02e9)
    assert bench.traffic_for("decode_kernel_512", "4bit", 2e9) is None
    assert bench.traffic_for("decode_kernel_512", "prefill", 1.0) is None


def test_cpu_sample_spreads_over_lengths():
    sys.path.insert(0, os.path.join(ROOT, "oracle"))
    import timing
    lengths = list(range(1000, 65000, 1000))
    idx = timing.sample_indices(lengths, 16)
    assert len(idx) == 16 and idx == sorted(idx)
    mean = sum(lengths[i] for i in idx) / 16
    assert abs(mean - sum(lengths) / len(lengths)) < 1000


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny", "--steps", "2", "--warmup", "3"], capture_output=True, text=True, cwd=ROOT,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 3 and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "2"],
                       capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_training_read_key_count_matches_the_oracle():
    """The flop count of the training-read workload counts exactly the keys
    the oracle's layout lets every row read."""
    import oracle as O
    for blocks in ([37, 20, 0, 9], [0, 5, 64], [70]):
        off = np.concatenate([[0], np.cumsum(blocks)])
        for window in (0, 1, 5, 100):
            want = sum(len(O.train_visible(off, r, window)) for r in range(int(off[-1])))
            assert bench.train_visible_total(blocks, window) == want

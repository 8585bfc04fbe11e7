"""Host-side pieces of bench.py, on CPU: the model FLOP count behind the MFU
figure (against the parameter layout), the clock sampler's reading of
nvidia-smi samples (median and maximum SM clock, every throttle reason seen
active), the roofline peaks (the measured file, else the stated fallback), and
the rule that a recorded DRAM traffic figure is reported only while the sources
it was captured on are unchanged."""
import hashlib
import importlib
import os
import stat
import time

import pytest

import bench
import oracle


@pytest.fixture
def fresh_bench():
    """bench with its module-level workload settings restored afterwards."""
    yield bench
    importlib.reload(bench)


# ----------------------------------------------------------------------------- FLOPs
@pytest.mark.parametrize("model", ["124m", "350m"])
def test_model_flops_per_token_counts_every_weight_matrix(fresh_bench, model):
    if model == "350m":
        fresh_bench.select_model("350m")
    b = fresh_bench
    sizes, _ = oracle.param_sizes(b.L, b.C, b.NH, b.V, b.Vp, b.MAXT)
    # the matrices every token multiplies by: qkvw, attprojw, fcw, fcprojw of each
    # layer, and the classifier over the V real vocabulary rows of wte
    qkvw, attprojw, fcw, fcprojw = sizes[4], sizes[6], sizes[10], sizes[12]
    n_matmul = qkvw + attprojw + fcw + fcprojw + b.V * b.C
    # forward 2 flops per weight, backward 4; causal attention: Q K^T and P V over
    # T/2 keys on average, forward and backward, 6 L C T in all
    want = 6.0 * n_matmul + 6.0 * b.L * b.C * b.T
    assert b.model_flops_per_token() == want
    if model == "124m":
        # 6.536 TFLOP per B=8, T=1024 step
        assert abs(want * b.B * b.T / 1e12 - 6.5357) < 1e-3


# ----------------------------------------------------------------------------- clocks
def _fake_smi(tmp_path, lines):
    d = tmp_path / "bin"
    d.mkdir()
    exe = d / "nvidia-smi"
    body = "\n".join(lines)
    # print the samples, then wait to be terminated like the real -lms loop
    exe.write_text(f"#!/bin/sh\ncat <<'END'\n{body}\nEND\nexec sleep 30\n")
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    return str(d)


def _sample(monkeypatch, path_dir, n_lines):
    monkeypatch.setenv("PATH", path_dir + os.pathsep + os.environ.get("PATH", ""))
    s = bench.ClockSampler(0)
    s.start()
    t0 = time.time()
    while time.time() - t0 < 10:
        with open(s.path) as f:
            if len(f.read().splitlines()) >= n_lines:
                break
        time.sleep(0.05)
    return s.stop()


def test_clock_sampler_reports_median_clock_and_power_cap(tmp_path, monkeypatch):
    lines = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1995, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 1390.2, 0x4, Not Active, Not Active, Not Active, Active",
             "0, [N/A], 2070, 1390.2, 0x0, Not Active, Not Active, Not Active, Not Active"]
    r = _sample(monkeypatch, _fake_smi(tmp_path, lines), len(lines))
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["samples"] == 3  # the unreadable sample is skipped
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_sampler_reports_slowdowns(tmp_path, monkeypatch):
    lines = ["0, 1410, 2070, 700.0, 0x8, Active, Not Active, Not Active, Not Active",
             "0, 1380, 2070, 690.0, 0x48, Not Active, Active, Active, Not Active",
             "0, 1500, 2070, 720.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    r = _sample(monkeypatch, _fake_smi(tmp_path, lines), len(lines))
    assert r["sm_mhz"] == 1410.0 and r["samples"] == 3
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    empty = tmp_path / "nothing"
    empty.mkdir()
    monkeypatch.setenv("PATH", str(empty))
    s = bench.ClockSampler(0)
    s.start()
    r = s.stop()
    assert r["sm_mhz"] is None and r["reasons"] == ["unavailable"]


# ----------------------------------------------------------------------------- peaks
def test_peaks_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback"
    assert (p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"]) == (6800.0, 1900.0, 1700.0)
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 7000.5, "bf16_tflops": 1950.0}')
    p = bench.load_peaks()
    assert p["source"] == "measured"
    # no sustained figure recorded: the burst one stands in for it
    assert (p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"]) == (7000.5, 1950.0, 1950.0)


# ----------------------------------------------------------------------------- traffic
def test_recorded_traffic_only_while_its_sources_are_unchanged(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "transformer_lm_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "a.cu").write_text("kernel a\n")
    (src / "b.cu").write_text("kernel b\n")
    h = hashlib.sha256(b"kernel a\nkernel b\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text(f"# capture\n\ntraffic_bytes: 123456\nsource_sha256_16: {h}\n")
    assert bench.profile_value("k.md", "traffic_bytes", ["a.cu", "b.cu"]) == 123456.0
    assert bench.profile_value("k.md", "other_key", ["a.cu", "b.cu"]) is None
    assert bench.profile_value("k.md", "traffic_bytes", ["b.cu", "a.cu"]) is None  # order matters
    assert bench.profile_value("missing.md", "traffic_bytes", ["a.cu", "b.cu"]) is None
    (src / "b.cu").write_text("kernel b, changed\n")
    assert bench.profile_value("k.md", "traffic_bytes", ["a.cu", "b.cu"]) is None

"""Host-side logic of bench.py (no GPU): the peak source, the traffic
figure's link to the kernel source, the workload description and the
CPU-baseline sample of the oracle."""
import hashlib
import json

import pytest

import bench


def test_fallback_peaks_without_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback"
    assert peaks["hbm_gbs"] == 6800.0 and peaks["bf16_tflops"] == 1900.0


def test_measured_peaks_are_found_by_key(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"gpu": {"hbm_gbs": 7100.5, "bf16_tflops": 2011.0}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "measured"
    assert bench._peak(peaks, "hbm_gbs") == 7100.5
    assert bench._peak(peaks, "bf16_tflops") == 2011.0
    assert bench._peak(peaks, "missing") is None


def test_traffic_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    src = tmp_path / "gemm_tc.cu"
    src.write_bytes(b"// kernel v1\n")
    prof = tmp_path / "profile.txt"
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    prof.write_text(f"# header\ngemm_tc.cu sha256: {sha}\ndram bytes per launch: 12345\n")
    monkeypatch.setattr(bench, "GEMM_SOURCE", str(src))
    monkeypatch.setattr(bench, "GEMM_PROFILE", str(prof))
    assert bench.gemm_traffic() == 12345.0
    src.write_bytes(b"// kernel v2\n")  # the kernel changed since the capture
    assert bench.gemm_traffic() is None
    monkeypatch.setattr(bench, "GEMM_PROFILE", str(tmp_path / "absent.txt"))
    assert bench.gemm_traffic() is None


def test_committed_profile_names_the_committed_kernel():
    """The committed ncu summary carries the hash of the kernel it measured;
    when the two agree the bench line reports the DRAM traffic."""
    with open(bench.GEMM_PROFILE) as f:
        text = f.read()
    assert "dram bytes per launch:" in text and "gemm_tc.cu sha256:" in text


def test_workload_matches_the_sweep():
    cfg = bench.config_dict()
    assert cfg["N"] == 10240 and cfg["K"] == 2560
    assert cfg["Ms"] == [1, 128, 1024, 4096, 8192]
    assert bench.step_ops() == pytest.approx(sum(2.0 * m * 10240 * 2560 for m in cfg["Ms"]))
    # the pages' per-channel sweep (Apple M5 Pro) as a whole-sweep rate
    assert bench.PAGES_TOPS == pytest.approx(
        bench.step_ops() / (sum(bench.PAGES_MS.values()) * 1e-3) / 1e12)


def test_oracle_sample_step_counts_the_rows_it_ran():
    import oracle
    oracle.build()
    inputs = bench.host_inputs()
    wq, sw = oracle.quantize_weight_int8(inputs["W"])
    inputs["wq_ref"], inputs["sw_ref"] = wq, sw
    ops, t = bench.oracle_sample_step(2, inputs)
    # two rows of every M except M = 1, which has one
    assert ops == pytest.approx(2.0 * 10240 * 2560 * (1 + 2 * 4))
    assert t > 0

"""Host-side helpers of bench.py (CPU only): the FLOP and byte counts behind the reported
rates, the peaks file, and the guard that keeps recorded DRAM traffic off a changed kernel."""
import json

import bench
from gen import make_decode


def test_prefill_flops_counts_visible_pairs():
    for S, causal in ((1, True), (7, True), (7, False), (130, True)):
        visible = sum(1 for i in range(S) for j in range(S) if (j <= i or not causal))
        assert bench.prefill_flops(2, 3, S, causal=causal) == 2.0 * 2 * 3 * visible * (192 + 128)
    # the headline workload's figure
    assert abs(bench.prefill_flops(4, 128, 4096) - 2.7495e12) < 1e9


def test_decode_kv_bytes_is_the_cache_the_lengths_need():
    inp = make_decode(3, 4, 1, [1, 64, 65], seed=3)
    assert bench.decode_kv_bytes(inp) == (1 + 64 + 65) * 576 * 2
    inp8 = make_decode(2, 4, 1, [10, 100], fp8=True, seed=4)
    assert bench.decode_kv_bytes(inp8) == (10 + 100) * (576 + 4)


def test_peaks_come_from_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks()["source"] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 2000.0}))
    pk = bench.peaks()
    assert pk["source"] == "measured" and pk["hbm_gbs"] == 7000.0 and pk["bf16_tflops"] == 2000.0


def test_recorded_traffic_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    csrc = tmp_path / "mla_flash_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_hash(["k.cu"])
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(
        json.dumps({"k": {"src_sha": sha, "dram_bytes_per_launch": 123.0}}))
    assert bench.recorded_traffic("k", ["k.cu"]) == 123.0
    (csrc / "k.cu").write_text("kernel v2")  # the kernel changed since the capture
    assert bench.recorded_traffic("k", ["k.cu"]) is None
    assert bench.recorded_traffic("missing", ["k.cu"]) is None

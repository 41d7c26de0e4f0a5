"""Host-side pieces of bench.py that need no GPU: the algorithmic byte counts
behind the roofline, the traffic record's source check, and the FP32 peak."""
import json

import bench
from sparse_head_self_gb300.inputs import WORKLOADS


def test_algorithmic_bytes_vitb():
    # B=64, H=12, N=197, D=64, bf16: forward reads Q, K, V and writes O (2 bytes
    # per element) plus one fp32 LSE per row; backward reads Q, K, V, O, dO and
    # LSE and writes dQ, dK, dV
    wl = WORKLOADS["vitb"]
    elems = 64 * 12 * 197 * 64
    rows = 64 * 12 * 197
    assert bench.algorithmic_bytes(wl, backward=False) == 4 * elems * 2 + 4 * rows == 78_068_736
    assert bench.algorithmic_bytes(wl, backward=True) == 8 * elems * 2 + 4 * rows == 155_532_288


def test_algorithmic_bytes_scale_with_dtype():
    wl = WORKLOADS["tiny"]   # fp32 rows
    elems = wl.B * wl.H * wl.N * wl.D
    rows = wl.B * wl.H * wl.N
    assert bench.algorithmic_bytes(wl, backward=False) == 4 * elems * 4 + 4 * rows


def test_traffic_record_follows_the_kernel_sources(monkeypatch, tmp_path):
    record = {"vitb": {"fibatt_bwd": {"dram_bytes_per_launch": 123, "source_hash": "abc"}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(record))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.recorded_traffic("fibatt_bwd", "vitb") == 123
    assert bench.recorded_traffic("fibatt_fwd", "vitb") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "changed")
    assert bench.recorded_traffic("fibatt_bwd", "vitb") is None


def test_committed_traffic_record_is_complete():
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        record = json.load(f)
    for workload in ("vitb", "video"):
        for kernel in ("fibatt_fwd", "fibatt_bwd"):
            ent = record[workload][kernel]
            assert ent["dram_bytes_per_launch"] > 0
            assert len(ent["source_hash"]) == 16


def test_fp32_peak():
    # 152 SMs x 128 FP32 lanes x 2 flops per FMA at 2070 MHz
    assert abs(bench.FP32_PEAK_TFLOPS - 80.54) < 0.01

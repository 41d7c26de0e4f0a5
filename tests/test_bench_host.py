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
    record = {"vitb": {"fibatt_bwd": {"dram_read": 100, "dram_write": 7, "l2_write": 30,
                                      "source_hash": "abc"}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(record))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    got = bench.recorded_traffic("fibatt_bwd", "vitb")
    # writes: the larger of the DRAM writes seen during the kernel and the
    # bytes written into L2 (dirty lines reach DRAM after the kernel ends)
    assert got["read"] == 100 and got["write"] == 30 and got["total"] == 130
    assert bench.recorded_traffic("fibatt_fwd", "vitb") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "changed")
    assert bench.recorded_traffic("fibatt_bwd", "vitb") is None


def test_committed_traffic_record_is_complete():
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        record = json.load(f)
    for workload, ents in record.items():
        assert workload in WORKLOADS
        for kernel, ent in ents.items():
            assert kernel in ("fibatt_fwd", "fibatt_bwd")
            assert ent["dram_read"] > 0 and ent["dram_write"] >= 0 and ent["l2_write"] > 0
            assert len(ent["source_hash"]) == 16


def test_roofline_record_picks_the_binding_roof():
    # vitb backward: 155.5 MB at 6783 GB/s (22.9 us) against 640 flops x 1.13 M
    # pairs at 80.5 TFLOP/s (9.0 us): HBM binds.  long backward: 539 MB (79.5 us)
    # against 640 x 12.7 M pairs (101 us): the FP32 units bind.
    vitb = bench.roofline_record(WORKLOADS["vitb"], "bwd", 0.05, 1_133_568, 6783.1, "measured")
    assert vitb["bound"] == "hbm"
    assert abs(vitb["GB_s"] - 155_532_288 / 0.05 / 1e6) < 0.1
    long_ = bench.roofline_record(WORKLOADS["long"], "bwd", 0.5, 12_710_168, 6783.1, "measured")
    assert long_["bound"] == "alu"
    assert abs(long_["TFLOP_s"] - 12_710_168 * 640 / 0.5e-3 / 1e12) < 0.01


def test_rotation_evicts_l2():
    l2 = 136 * 2**20
    assert bench._rotation(166_000_000, l2) == 4            # vitb sets
    assert bench._rotation(650_000_000, l2) == 2            # long sets: larger than L2 each
    assert bench._rotation(200_000, l2) == 64               # tiny: capped


def test_fp32_peak():
    # 152 SMs x 128 FP32 lanes x 2 flops per FMA at 2070 MHz
    assert abs(bench.FP32_PEAK_TFLOPS - 80.54) < 0.01

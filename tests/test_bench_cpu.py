"""bench.py's bookkeeping on the host (no GPU): the algorithmic bytes of the coarse pass, the
roofline bound it reports, and the rule that a recorded DRAM traffic figure is used only while
the kernel sources it was taken on are unchanged."""
import hashlib
import json
import os

import bench


def test_algorithmic_bytes_of_the_full_and_shard_heads():
    # packed V*H/4 plus S and ZS (two bf16 per row and group of 128)
    assert bench.algorithmic_bytes(248320, 5120) == 248320 * 1280 + 2 * 248320 * 40 * 2
    assert bench.algorithmic_bytes(248320, 5120) == 357_580_800
    assert bench.algorithmic_bytes(124160, 5120) == 178_790_400
    assert bench.algorithmic_bytes4(248320, 5120) == 248320 * 2560 + 2 * 248320 * 40 * 2


def test_roofline_entry_picks_the_longer_bound():
    # M=16: the weight stream (357.6 MB at 6780 GB/s = 52.7 us) dwarfs 40.7 GFLOP at the bf16 peak
    r = bench.roofline_entry(16, 110.8, 6780.0, 1928.0, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 357_580_800 / 110.8 / 1e3) < 0.1
    assert abs(r["frac"] - r["achieved"] / 6780.0) < 1e-4
    # M=32 is still the weight stream's (81.4 GFLOP / 1928 TF/s = 42.2 us < 52.7 us) ...
    assert bench.roofline_entry(32, 160.0, 6780.0, 1928.0, "measured")["bound"] == "hbm"
    # ... and M=64 the contraction's, against the bf16 peak itself (162.7 GFLOP -> 84.4 us)
    r = bench.roofline_entry(64, 320.0, 6780.0, 1928.0, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1928.0
    assert abs(r["achieved"] - 2 * 64 * 5120 * 248320 / 320.0 / 1e6) < 0.1
    assert abs(r["frac"] - r["achieved"] / 1928.0) < 1e-4
    # the one-shard head: half the bytes and flops
    r = bench.roofline_entry(16, 60.0, 6780.0, 1928.0, "measured", V=124160)
    assert r["bytes_per_launch"] == 178_790_400


def test_recorded_traffic_is_dropped_once_a_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("__global__ void k() {}\n")
    rec = {"sources": ["kernel.cu"], "traffic_per_launch": {"16": 123},
           "sha256": hashlib.sha256(src.read_bytes()).hexdigest()}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "coarse_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile(16) == 123
    assert bench.traffic_from_profile(32) is None
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.traffic_from_profile(16) is None


def test_committed_traffic_record_names_existing_sources():
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "coarse_traffic.json")))
    assert rec["sources"] and all(os.path.exists(os.path.join(bench.ROOT, f)) for f in rec["sources"])
    per = rec["traffic_per_launch"]["16"]
    assert 1.0 <= per / bench.algorithmic_bytes(248320, 5120) < 1.1

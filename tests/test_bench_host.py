"""Host-side logic of bench.py that needs no GPU: the committed DRAM-traffic
records behind roofline.traffic (reported only while the GEMM sources hash to
the value a record was captured with) and the roofline denominators."""
import glob
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from w8a8_int8_linear_gb300 import workloads as wl  # noqa: E402

REQUIRED = ("workload", "kernel", "gemm_source_sha256_16", "dram_bytes_read", "dram_bytes_write")


def _records():
    return sorted(glob.glob(os.path.join(ROOT, "profiles", "gemm_traffic_*.txt")))


def _parse(path):
    kv = {}
    for line in open(path):
        if "=" in line and not line.lstrip().startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    return kv


def test_traffic_records_are_complete():
    paths = _records()
    assert paths, "no traffic record under profiles/"
    for p in paths:
        kv = _parse(p)
        for k in REQUIRED:
            assert k in kv, f"{os.path.basename(p)}: {k} missing"
        assert kv["workload"] in wl.ALL, kv["workload"]
        assert os.path.basename(p) == f"gemm_traffic_{kv['workload']}.txt"
        assert int(kv["dram_bytes_read"]) > 0 and int(kv["dram_bytes_write"]) > 0
        assert len(kv["gemm_source_sha256_16"]) == 16
        if "scale_to_full" in kv:
            work = wl.ALL[kv["workload"]]
            assert float(kv["scale_to_full"]) == work.M / int(kv["captured_M"])


def test_gemm_source_hash_covers_the_listed_sources():
    for f in bench.GEMM_SOURCES:
        assert os.path.exists(os.path.join(ROOT, "w8a8_int8_linear_gb300", "csrc", f)), f
    h = bench.gemm_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert bench.gemm_source_hash() == h


@pytest.mark.parametrize("path", _records(), ids=os.path.basename)
def test_recorded_traffic_follows_the_source_hash(monkeypatch, path):
    kv = _parse(path)
    work = kv["workload"]
    scale = float(kv.get("scale_to_full", "1"))
    expect = (int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])) * scale
    # sources as captured: the record's bytes, scaled to the full launch
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: kv["gemm_source_sha256_16"])
    t, how = bench.recorded_traffic(work)
    assert t == expect and os.path.basename(path) in how
    # any other source state: no traffic claimed
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 16)
    t, how = bench.recorded_traffic(work)
    assert t is None and "changed" in how


def test_recorded_traffic_without_a_record():
    t, how = bench.recorded_traffic("tiny_postscale_64x128x256")
    assert t is None and "no record" in how


def test_peaks_from_the_measured_file_or_the_fallback(tmp_path, monkeypatch):
    p = bench.load_peaks()
    assert p["hbm_gbs"] > 0 and p["bf16_tflops"] > 0 and p["bf16_tflops_sustained"] > 0
    measured = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(measured):
        d = json.load(open(measured))
        assert p["source"] == "measured" and p["hbm_gbs"] == float(d["hbm_gbs"])
    # a tree without the file: the fallback figures
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = bench.load_peaks()
    assert f["source"] == "fallback"
    assert (f["hbm_gbs"], f["bf16_tflops"]) == (bench.FALLBACK_HBM_GBS, bench.FALLBACK_BF16_TFLOPS)

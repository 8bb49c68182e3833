"""Host logic of bench.py that needs no GPU: the committed DRAM-traffic figure
is reported only for the decode source it was measured on, and nvidia-smi
clock samples are summarised into the median clock and the throttle reasons
seen."""
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_traffic_only_for_the_measured_decode_source(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "decode_traffic.json")))
    fake = tmp_path / "repo"
    (fake / "profiles").mkdir(parents=True)
    csrc = fake / "quantized_attention_kv_b300" / "csrc"
    csrc.mkdir(parents=True)
    srcs = {n: open(os.path.join(ROOT, "quantized_attention_kv_b300", "csrc", n)).read()
            for n in bench.DECODE_SOURCES}
    for n, t in srcs.items():
        (csrc / n).write_text(t)
    rec["decode_sources_sha256_16"] = bench.decode_source_hash(str(fake))
    (fake / "profiles" / "decode_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(fake))
    assert bench._traffic(1) == rec["dram_bytes_per_call"]
    for n in bench.DECODE_SOURCES:                                # any of them changed since
        (csrc / n).write_text(srcs[n] + "\n// changed\n")
        assert bench._traffic(1) is None, n
        (csrc / n).write_text(srcs[n])
        assert bench._traffic(1) == rec["dram_bytes_per_call"]


def test_clock_summary(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text(
        "0, 2032, 2032, 812.40, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "0, 1980, 2032, 1093.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
        "0, 2010, 2032, 1001.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "garbage line\n")
    cs = bench.ClockSampler(0)
    cs.path = str(path)
    s = cs.summary()
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2032 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    cs.path = str(tmp_path / "missing.csv")
    assert cs.summary()["reasons"] == ["no samples"]

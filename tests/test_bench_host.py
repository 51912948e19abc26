"""Host-side logic of bench.py that decides what its JSON line reports (CPU).

- ClockSampler.summary: the median SM clock under load (idle samples below
  30 % of the maximum left out), the maximum clock, the throttle reasons seen
  active and the peak power, from nvidia-smi's CSV rows.
- recorded_traffic: the committed ncu DRAM bytes are reported only while the
  kernel sources hash to the value recorded with them; a stale or malformed
  record gives None (roofline.traffic null).
- load_peaks: the measured peaks file, else the fallback figures, labelled.
- workload_config: the workload's description, without implementation keys.
"""
import os

import pytest

import bench
from recommender_attention_gb300 import workloads as W


def _row(sm, smax, power, active=("Not Active",) * 4):
    return ", ".join(["0", str(sm), str(smax), str(power), "0x0000000000000000", *active])


def _summary_of(tmp_path, rows):
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler(0)
    s.proc = object()          # a sampler that ran; only its CSV is read
    s.path = str(path)
    out = s.summary()
    assert not path.exists(), "the summary removes its sample file"
    return out


def test_clock_summary_median_under_load_and_reasons(tmp_path):
    rows = [_row(345, 2070, 150.0),                                   # idle before the timed region
            _row(1800, 2070, 1100.5),
            _row(1830, 2070, 1350.0, ("Not Active", "Not Active", "Not Active", "Active")),
            _row(1860, 2070, 1390.25),
            _row(120, 2070, 90.0)]                                   # idle after it
    out = _summary_of(tmp_path, rows)
    assert out["sm_mhz"] == 1830.0          # median of the three samples above 30 % of 2070
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 5
    assert out["power_w_max"] == 1390.25


def test_clock_summary_reports_every_slowdown_kind(tmp_path):
    rows = [_row(1500, 2070, 900, ("Active", "Not Active", "Not Active", "Not Active")),
            _row(1400, 2070, 900, ("Not Active", "Active", "Active", "Not Active"))]
    out = _summary_of(tmp_path, rows)
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1450.0


def test_clock_summary_without_samples(tmp_path):
    assert _summary_of(tmp_path, [])["reasons"] == ["no samples"]
    s = bench.ClockSampler(0)
    assert s.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    rec = tmp_path / "dram.txt"
    good = bench.kernel_source_hash()
    rec.write_text("# a comment: with a colon\n"
                   f"kernel_source_hash: {good}\n"
                   "dram_bytes_read: 600\n"
                   "dram_bytes_write: 100\n"
                   "dram_bytes_per_launch: 700\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.recorded_traffic() == 700
    rec.write_text(rec.read_text().replace(good, "0123456789abcdef"))
    assert bench.recorded_traffic() is None, "a record of other kernel sources must not be reported"
    rec.write_text(f"kernel_source_hash: {good}\n")
    assert bench.recorded_traffic() is None, "a record without the byte count"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.txt"))
    assert bench.recorded_traffic() is None


def test_committed_traffic_record_is_well_formed():
    """The committed record parses and its bytes add up; whether it matches the
    current sources is what recorded_traffic checks at run time."""
    kv = {}
    with open(bench.TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    assert len(kv["kernel_source_hash"]) == 16
    assert int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"]) == int(kv["dram_bytes_per_launch"])


def test_load_peaks_fallback(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "PEAKS_FILE", str(tmp_path / "absent.json"))
    peaks, kind = bench.load_peaks()
    assert kind == "fallback"
    assert peaks == bench.FALLBACK_PEAKS and peaks is not bench.FALLBACK_PEAKS
    f = tmp_path / "peaks.json"
    f.write_text('{"hbm_gbs": 6000.0, "bf16_tflops": 1900.0}')
    monkeypatch.setattr(bench, "PEAKS_FILE", str(f))
    peaks, kind = bench.load_peaks()
    assert kind == "measured" and peaks["hbm_gbs"] == 6000.0


@pytest.mark.parametrize("world", [1, 4])
def test_workload_config_describes_the_workload_only(world):
    w = W.large_jagged(hdim=128)
    c = bench.workload_config(w, allowed_pairs=12345, world=world)
    assert c["batch"] == w.batch and c["nhead"] == w.nhead and c["total_tokens"] == w.total_q
    assert c["allowed_pairs"] == 12345
    assert c["parallelism"] == ("single GPU" if world == 1 else f"replicas x{world}")
    for key in ("num_splits", "executed_tiles", "model", "cta_pairs"):
        assert key not in c

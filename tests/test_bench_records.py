"""bench.py's host-side records, no GPU needed: the roofline `traffic` comes from a committed
ncu record only when that record was taken on the current kernel source and on the same
workload, and the `clocks` summary keeps the nvidia-smi samples of the timed region (or the
nearest one) with their throttle reasons."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_records_match_their_sources_and_workloads():
    for record, source, workload in (("decode_attention_traffic.json", "decode_attention.cu", "bandwidth"),
                                     ("prefill_attention_traffic.json", "prefill_attention.cu", "prefill")):
        with open(os.path.join(ROOT, "profiles", record)) as f:
            rec = json.load(f)
        assert rec["traffic_bytes_per_launch_full_workload"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        with open(os.path.join(ROOT, "paged_kv_cache_180_gb300", "csrc", source), "rb") as f:
            current = hashlib.sha256(f.read()).hexdigest() == rec["kernel_source_sha256"]
        got = bench.committed_traffic(record, source, workload)
        # the figure is reported only while the record matches the kernel source
        assert got == (rec["traffic_bytes_per_launch_full_workload"] if current else None)
        # another workload, or a record of another source, gives no traffic figure
        assert bench.committed_traffic(record, source, "ragged") is None
        other = "prefill_attention.cu" if source == "decode_attention.cu" else "decode_attention.cu"
        assert bench.committed_traffic(record, other, workload) is None


def test_nvtx_ranges_are_off_by_default():
    assert bench.NVTX is False
    with bench.nvtx("anything"):
        pass


def _smi_line(sm, mx, power, hw="Not Active", thermal="Not Active", sw_thermal="Not Active", cap="Not Active"):
    # the fields of ClockSampler.QUERY, in order, as nvidia-smi prints them (csv, no units)
    return f"2026/01/01 00:00:00.000, 0, {sm}, {mx}, {power}, 0x0000000000000000, {hw}, {thermal}, {sw_thermal}, {cap}"


def test_clock_summary_takes_the_samples_inside_the_timed_region():
    s = bench.ClockSampler(0)
    s.lines = [(9.0, _smi_line(1000, 2070, 100.0, hw="Active")),      # before the region: ignored
               (10.0, _smi_line(2070, 2070, 600.0)),
               (10.1, _smi_line(2040, 2070, 700.0, cap="Active")),
               (10.2, _smi_line(2055, 2070, 650.0)),
               (12.0, _smi_line(500, 2070, 90.0, thermal="Active"))]  # after it: ignored
    out = s.summary(10.0, 10.2)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 700.0


def test_clock_summary_reports_slowdowns_and_falls_back_to_the_nearest_sample():
    s = bench.ClockSampler(0)
    s.lines = [(5.0, _smi_line(1500, 2070, 300.0, hw="Active", sw_thermal="Active")), (7.0, "garbled line")]
    inside = s.summary(5.0, 5.001)
    assert inside["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and inside["samples"] == 1
    near = s.summary(5.2, 5.203)  # shorter than the sampling period, no sample inside
    assert near["samples"] == 1 and near["sm_mhz"] == 1500.0 and "note" in near
    assert bench.ClockSampler(0).summary(0.0, 1.0)["samples"] == 0


def test_prefill_shape_option_names_its_workload():
    import types
    assert bench.prefill_shape(types.SimpleNamespace(prefill_shape="16,512")) == (16, 512, "prefill")
    assert bench.prefill_shape(types.SimpleNamespace(prefill_shape="4,2048")) == (4, 2048, "prefill_4x2048")
    assert bench.prefill_shape(types.SimpleNamespace()) == (16, 512, "prefill")
    # a shape other than the recorded one never picks up the committed traffic record
    assert bench.committed_traffic("prefill_attention_traffic.json", "prefill_attention.cu", "prefill_4x2048") is None

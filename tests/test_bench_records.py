"""bench.py's roofline `traffic` comes from a committed ncu record only when that record was
taken on the current kernel source and on the same workload (no GPU needed)."""
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

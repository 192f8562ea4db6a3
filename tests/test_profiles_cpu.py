"""The committed DRAM-traffic captures belong to the kernel sources in the tree.

bench.py reports a kernel's measured DRAM traffic only from a profiles/traffic.json
entry whose source hash equals that of the kernel's current sources, and reports
null otherwise. A kernel change without a new capture would therefore turn the
benchmark line's traffic into null without any error; this test catches it first.
"""
import json

import bench

WORKLOADS = ["mxfp8_prefill_zipf", "mxfp8_small", "nvfp4_decode", "nvfp4_shared_norm", "mxfp4_small"]


def test_traffic_entries_match_kernel_sources():
    doc = json.load(open(bench.TRAFFIC_FILE))
    sha = bench.kernel_source_hash("mlp")
    entries = [e for e in doc["entries"] if e["kernel"] == "mlp"]
    stale = sorted(e["workload"] for e in entries if e["source_sha"] != sha)
    assert not stale, f"traffic captured from other GEMM sources (current {sha}): {stale}"
    assert sorted(e["workload"] for e in entries) == sorted(WORKLOADS)
    for e in entries:
        assert e["dram_bytes_per_launch"] > 0
        assert "--clock-control none" in e["command"]


def test_bench_uses_the_entries():
    for w in WORKLOADS:
        value, source = bench.measured_traffic(w, "mlp")
        assert value is not None and value > 0, source

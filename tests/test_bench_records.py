"""bench.py's use of the committed ncu records: traffic is reported only for the workload a
capture was taken on, and only while the kernel's code (not its comments) is unchanged."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_records_resolve_only_for_their_workload():
    recs = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    assert set(recs) <= set(bench.KERNEL_SOURCES)
    for kernel, e in recs.items():
        got = bench.recorded_traffic(kernel, e["workload"])
        if got is not None:  # current sources: the recorded bytes
            assert got == int(e["dram_bytes_per_launch"])
        assert bench.recorded_traffic(kernel, e["workload"] + "_other") is None


def test_code_hash_ignores_comments_not_code():
    src = "int f(int x) {  // doubles\n  /* the body */ return 2 * x;\n}\n"
    same = "int f(int x) {  // twice\n  return 2 *   x;\n}\n"
    other = "int f(int x) {  // doubles\n  return 3 * x;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)

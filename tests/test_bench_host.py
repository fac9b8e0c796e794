"""bench.py host logic that needs no GPU: the recorded-traffic bookkeeping."""
import json
import os

import bench


def test_code_only_drops_comments_not_code():
    src = 'int a = 1;  // one\n// a whole comment line\n\nconst char* s = "x // y";  // tail\n'
    got = bench._code_only(src)
    assert got == 'int a = 1;\nconst char* s = "x // y";'
    # a comment edit keeps the code, a code edit changes it
    assert bench._code_only(src.replace("// one", "// uno")) == got
    assert bench._code_only(src.replace("= 1", "= 2")) != got


def test_recorded_traffic_entries_are_well_formed():
    path = os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")
    t = json.load(open(path))
    for kernel, per_workload in t.items():
        for workload, e in per_workload.items():
            assert e["bytes_per_launch"] == e["read"] + e["write"], (kernel, workload)
            assert len(e["source_hash"]) == 16 and e["note"]
            # reported only while the kernel's code matches the capture
            got = bench.recorded_traffic(kernel, workload)
            assert got is None or got == float(e["bytes_per_launch"])

"""Host-side pieces of the benchmark that decide what its JSON line reports
(no GPU): which calls enter the roofline figure of a sweep, and that every
workload's dominant kernel has a DRAM traffic record to report."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _traffic_rows():
    rows = {}
    for line in open(os.path.join(ROOT, "profiles", "dram_traffic.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, src, digest, per_launch = line.split()[:4]
        rows[name] = (src, digest, int(per_launch))
    return rows


def test_every_workload_kernel_has_a_traffic_row():
    rows = _traffic_rows()
    for name, cls in bench.WORKLOADS.items():
        assert cls.kernel in rows, (name, cls.kernel)
        src = rows[cls.kernel][0]
        assert os.path.exists(os.path.join(ROOT, "weight_only_bit_split_gb300", "csrc", src))
        assert rows[cls.kernel][2] > 0


def test_traffic_record_needs_the_recorded_source():
    rows = _traffic_rows()
    for kernel, (src, digest, per_launch) in rows.items():
        got = bench.traffic_record(kernel)
        assert got is None or got == float(per_launch)
    assert bench.traffic_record("no_such_kernel") is None


def test_sweeps_report_their_dominant_kernel_only():
    q4 = bench.Q4Sweep
    assert q4.kernel == "q4_0_q8_1_mma"
    dominant = [f"M{m}_{n}x{k}" for m in q4.Ms for n, k in q4.shapes if q4.roofline_call(f"M{m}_{n}x{k}")]
    assert sorted({int(x[1:].split("_")[0]) for x in dominant}) == [8, 12, 16]
    nf4 = bench.NF4Sweep
    assert nf4.kernel == "nf4_tc"
    assert not any(nf4.roofline_call(f"M{m}") for m in nf4.Ms if m <= 4)
    assert all(nf4.roofline_call(f"M{m}") for m in nf4.Ms if m > 4)


def test_every_environment_knob_is_documented():
    """Each WOBS_* variable the library reads is described in the header."""
    import re
    csrc = os.path.join(ROOT, "weight_only_bit_split_gb300", "csrc")
    names = set()
    for f in os.listdir(csrc):
        if f.endswith((".cu", ".cuh", ".h")):
            names |= set(re.findall(r'getenv\("(WOBS_[A-Z0-9_]+)"\)', open(os.path.join(csrc, f)).read()))
    header = open(os.path.join(ROOT, "include", "wobs.h")).read()
    assert names and all(n in header for n in names), sorted(n for n in names if n not in header)

"""The committed ncu summaries and the benchmark that reads them (CPU only).

bench.py takes a launch's DRAM traffic from the summary of its workload
(profiles/*_step_<workload>.md) only while the summary's source digest matches
the kernel sources it was captured on; these tests hold the summaries to the
fields that rule needs and to the kernel the benchmark says it times.
"""
import glob
import os
import re

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAMILY_KERNEL = {"decode": "decode_kernel", "mixed": "mixed_kernel", "decode_tc": "decode_tc_kernel",
                 "decode_tc8": "decode_tc8_kernel", "prefill_tc": "prefill_tc_kernel"}


def _fields(path):
    out = {}
    for line in open(path):
        m = re.match(r"<!-- (\w+): (.*) -->", line.strip())
        if m:
            out[m.group(1)] = m.group(2).strip()
    return out


def _summaries():
    return sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def test_every_summary_names_workload_family_digest_and_traffic():
    paths = _summaries()
    assert paths
    for p in paths:
        f = _fields(p)
        assert {"workload", "kernel_family", "source_sha", "dram_bytes_per_launch"} <= set(f), p
        assert f["kernel_family"] in bench.KERNEL_SOURCES, p
        assert re.fullmatch(r"[0-9a-f]{16}", f["source_sha"]), p
        assert int(f["dram_bytes_per_launch"]) > 0, p
        text = open(p).read()
        assert "--clock-control none" in text, f"{p}: an ncu command without --clock-control none"


def test_step_summaries_describe_the_kernel_the_benchmark_times():
    for p in _summaries():
        if "_step_" not in os.path.basename(p):
            continue
        f = _fields(p)
        w = synth.make_workload(f["workload"], seed=0)
        assert FAMILY_KERNEL[f["kernel_family"]] in bench.step_kernel(w), (p, bench.step_kernel(w))


def test_traffic_is_read_only_from_a_current_summary():
    """profiled_traffic gives the summary's bytes when its digest matches the sources, else nothing."""
    for p in _summaries():
        if "_step_" not in os.path.basename(p):
            continue
        f = _fields(p)
        got = bench.profiled_traffic(f["workload"])
        if f["source_sha"] == bench.source_digest(f["kernel_family"]):
            assert got == int(f["dram_bytes_per_launch"]), p
        else:
            assert got is None, p

"""Host-side pieces of bench.py: the profile summaries it reads the DRAM traffic from."""
from __future__ import annotations

import glob
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_profile_fields_keeps_colons_in_keys():
    text = "# title\n- gemm.cu sha256[:16]: `abc123`\n- dram bytes per launch: `42`\nnot a field: x\n"
    assert bench.profile_fields(text) == {"gemm.cu sha256[:16]": "abc123",
                                          "dram bytes per launch": "42"}


def test_committed_traffic_summaries_parse():
    paths = glob.glob(os.path.join(ROOT, "profiles", "traffic_*_kernel_*.md"))
    assert paths
    for p in paths:
        vals = bench.profile_fields(open(p).read())
        assert len(vals["gemm.cu sha256[:16]"]) == 16
        assert int(vals["dram bytes per launch"]) > 0
        kernel, workload = os.path.basename(p)[len("traffic_"):-len(".md")].split("_kernel_")
        got = bench.recorded_traffic(kernel, workload)
        if vals["gemm.cu sha256[:16]"] == bench.kernel_source_hash():
            assert got == float(vals["dram bytes per launch"])
        else:
            assert got is None     # counters taken on another version of the kernel

"""Host-side pieces of bench.py: the profile summaries it reads the DRAM traffic from."""
from __future__ import annotations

import glob
import os

import bench
import synth

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


def test_algorithmic_bytes_by_activation_format():
    w = synth.WORKLOADS["layer_T512"]
    ids, _ = synth.routing(w)
    a4 = bench.algorithmic(w, ids)
    a8 = bench.algorithmic(w, ids, act_fp8=True)
    A = w.T * w.k
    # same weights and FLOPs; the E4M3 token rows take H/2 more bytes each
    assert a8["flops"] == a4["flops"] == 6 * A * w.H * w.I
    assert a8["layer_kernel_bytes"] - a4["layer_kernel_bytes"] == A * (w.H // 2)
    assert a4["layer_kernel_bytes"] == 256 * 13369344 + A * 2176

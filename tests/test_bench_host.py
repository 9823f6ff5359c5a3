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


def test_vs_baseline_only_where_the_pages_give_a_figure():
    """vs_baseline divides by the pages' own tokens/s for the same layer (512 tokens in
    537.6 us for W4A4, 753.2 us for W4A8, one rank); null for other workloads, formats,
    GPU counts or overridden sizes."""
    class Args:
        mma, tokens, experts = "mxf4xmxf4", 0, 0

    a = Args()
    t512 = synth.WORKLOADS["layer_T512"]
    r, basis = bench.pages_ratio(a, t512, 1, 512 / 537.6e-6)
    assert abs(r - 1.0) < 1e-12 and "537.6" in basis and "B200" in basis
    a.mma = "fp8xfp4"
    r, _ = bench.pages_ratio(a, t512, 1, 2 * 512 / 753.2e-6)
    assert abs(r - 2.0) < 1e-12
    a.mma = "nvf4xnvf4"
    assert bench.pages_ratio(a, t512, 1, 1e6) == (None, None)
    a.mma = "mxf4xmxf4"
    assert bench.pages_ratio(a, synth.WORKLOADS["prefill_T4096"], 1, 1e6) == (None, None)
    assert bench.pages_ratio(a, t512, 2, 2e6) == (None, None)
    a.tokens = 256
    assert bench.pages_ratio(a, t512, 1, 1e6) == (None, None)

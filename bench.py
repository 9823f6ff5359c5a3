"""Benchmark of the W4A4 MXFP4 mixture-of-experts layer on GB300.

One step = one pass of the whole layer (moe_pre_dispatch + moe_forward) over one batch
of synthetic tokens: quantise + bucket, gate/up GEMM + SwiGLU + requantisation, down
GEMM + top-k weighted combine.  Default workload: the DeepSeek-V4-Flash layer at
T=512 tokens (hidden 4096, inter 2048, 256 experts, top-6), the point the pages
measure in isolation ("[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4 mega-MoE
(W4A4)", Appendix B).

Prints one JSON line.  `value` is tokens/s of the whole job (all ranks) with inputs
resident in HBM; `e2e` is the same metric through moe_run_host on pinned host buffers
(copies included); `roofline` is the dominant kernel's achieved HBM bandwidth against
the measured copy peak; `cpu_baseline` times the CPU oracle on a bounded sample.
--impl reference times the CPU oracle as the reference arm.
Multi-GPU (torchrun): independent replicas, one per GPU (the layer does not shard here).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_FLUSH_BYTES = 512 << 20          # > 2x the 129 MB L2
L2_CLEAN_BYTES = 256 << 20          # read after the write flush, so that its dirty
                                    # lines are written back before the timed step
KERNELS_PER_STEP = 4                # bucket, quantize_scatter, layer (both GEMMs + combine), convert
METRIC = "W4A4 MoE layer tokens/s (E=256, top-6, T=512; also us/layer and HBM TB/s)"
METRIC_W4A8 = "W4A8 (fp8xfp4) MoE layer tokens/s (E=256, top-6, T=512; also us/layer and HBM TB/s)"
METRIC_NVF4 = "NVFP4 (nvf4xnvf4) MoE layer tokens/s (E=256, top-6, T=512; also us/layer and HBM TB/s)"


def w4a8(args) -> bool:
    """fp8xfp4: MXFP8 activations against the same MXFP4 weights."""
    return args.mma == "fp8xfp4"


def nvf4(args) -> bool:
    """nvf4xnvf4: NVFP4 weights and activations (E4M3 scale per 16 elements)."""
    return args.mma == "nvf4xnvf4"


def metric(args) -> str:
    return METRIC_W4A8 if w4a8(args) else METRIC_NVF4 if nvf4(args) else METRIC


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="layer_T512", choices=sorted(synth.WORKLOADS))
    p.add_argument("--experts", type=int, default=0,
                   help="override the expert count (small cases for profiler captures)")
    p.add_argument("--tokens", type=int, default=0, help="override the token count")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--dispatch", choices=["bucketed", "pull"], default="bucketed",
                   help="token rows copied per expert by pre_dispatch, or gathered by the layer")
    p.add_argument("--tiles", choices=["auto", "wide", "medium", "narrow", "pair"], default="auto",
                   help="token tiles: 128 rows (wide), 64 (medium), 32 (narrow), 192 on SM pairs "
                        "(pair) or the layer's choice")
    p.add_argument("--mma", choices=["mxf4xmxf4", "fp8xfp4", "nvf4xnvf4"], default="mxf4xmxf4",
                   help="formats: MXFP4 (W4A4, the headline), MXFP8 activations (W4A8) or NVFP4")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other DeepSeek-V4-Flash configurations (the `workloads` object)")
    p.add_argument("--cpu-sample-tokens", type=int, default=0)
    return p.parse_args()


def workload(args) -> synth.Workload:
    w = synth.WORKLOADS[args.workload]
    if args.experts or args.tokens:
        E = args.experts or w.E
        T = args.tokens or w.T
        w = synth.Workload(f"{w.name}_T{T}_E{E}", T=T, H=w.H, I=w.I, E=E, k=min(w.k, E),
                           routing=w.routing, zipf_s=w.zipf_s, outlier_frac=w.outlier_frac)
    return w


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------
# Clock sampling during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval_ms = interval_ms   # short: the timed passes last tens of milliseconds
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms), "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Algorithmic bytes and FLOPs

def touched_experts(ids, E):
    return int(np.count_nonzero(np.bincount(ids.reshape(-1), minlength=E)))


def algorithmic(w: synth.Workload, ids, act_fp8: bool = False, sf_group: int = 32) -> dict:
    """Bytes a perfect implementation must move, and FLOPs.  act_fp8: the token rows
    are E4M3 (one byte an element) instead of packed E2M1; sf_group: elements per
    scale byte (16 for NVFP4)."""
    H, I, k, T = w.H, w.I, w.k, w.T
    A = T * k
    u = touched_experts(ids, w.E)
    w1 = 2 * I * H // 2 + 2 * I * H // sf_group     # gate/up codes + scales per expert
    w2 = H * I // 2 + H * I // sf_group             # down codes + scales per expert
    return {
        "touched_experts": u,
        "layer_bytes": u * (w1 + w2) + 2 * T * H + 2 * T * H + 8 * T * k,
        # layer kernel: every touched expert's weights and the quantised token rows it
        # reads once
        "layer_kernel_bytes": u * (w1 + w2) + A * ((H if act_fp8 else H // 2) + H // sf_group),
        "flops": 6 * A * H * I,
    }


# The part's nominal HBM3e bandwidth (GB/s), the denominator the target at T=512 names
# (>= 75% of about 8 TB/s); reported beside the fraction of the measured copy peak.
NOMINAL_HBM_GBS = 8000.0
# The DeepSeek-V4-Flash configurations besides the headline one, measured on the same
# prepared weights (they share H, I and E) and reported in the `workloads` object.
OTHER_WORKLOADS = ("decode_T64", "prefill_T4096", "prefill_T16384_zipf")

# Nominal dense FP4 : bf16 tensor throughput of the part (13.5 : 2.25 PFLOP/s), and
# FP8 : bf16 (4.5 : 2.25) for the fp8xfp4 MMAs (kind::mxf8f6f4 runs at the FP8 rate).
FP4_PER_BF16 = 6.0
FP8_PER_BF16 = 2.0


# The pages' own layer times for the benchmark's workload (the DeepSeek-V4-Flash layer at
# ntok=512, one rank in isolation; "[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4
# mega-MoE (W4A4)", Appendix B), measured on B200: context for the ratio, not a target.
PAGES_US_T512 = {"mxf4xmxf4": 537.6, "fp8xfp4": 753.2}


def pages_ratio(args, w, world: int, value: float):
    """value / the pages' tokens/s for the same workload and mma type on one GPU, and
    what the ratio is against; (None, None) where the pages give no figure."""
    us = PAGES_US_T512.get(args.mma)
    if us is None or w.name != "layer_T512" or world != 1 or args.tokens or args.experts:
        return None, None
    ref = w.T / (us * 1e-6)
    return value / ref, (f"the pages' {us} us per layer ({ref:.0f} tokens/s) for this layer at "
                         "ntok=512, one rank, measured on B200 (another GPU: context)")


def fp4_peak_from_bf16(peaks: dict) -> float:
    """The FP4 tensor peak in TFLOP/s: the measured bf16 GEMM peak (burst: the layer
    kernel is timed alone, for well under a second) times the nominal FP4:bf16 ratio."""
    return float(peaks["bf16_tflops"]) * FP4_PER_BF16


def fp4_mma_probe(mx, ws, stream, n_sms: int) -> dict:
    """FP4 tensor throughput measured with the library's MMA probe (operands in
    shared memory, no global traffic), per tile shape; best of three launches."""
    import torch

    out = {}
    count = 1 << 18

    def best_ms(launch):
        best = float("inf")
        with torch.cuda.stream(stream):
            launch()
            for _ in range(3):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                launch()
                b.record(stream)
                b.synchronize()
                best = min(best, a.elapsed_time(b))
        mx.moe_check(ws, stream)
        return best

    # single-CTA M=128 forms (2 or 1 blocks an SM)
    for n, bps in ((128, 2), (256, 1)):
        blocks = n_sms * bps
        ms = best_ms(lambda: mx.moe_fp4_mma_probe(ws, n, bps, blocks, count, stream))
        out[f"n{n}_x{bps}"] = blocks * count * 2.0 * 128 * n * 64 / (ms / 1e3) / 1e12
    # the two-SM M=256 form (cta_group::2), one pair of CTAs per two SMs
    pairs = n_sms // 2
    for n in (256,):
        ms = best_ms(lambda: mx.moe_fp4_mma_probe_pair(ws, n, pairs, count, stream))
        out[f"m256_n{n}_pair"] = pairs * count * 2.0 * 256 * n * 64 / (ms / 1e3) / 1e12
    return out


def mxfp8_producer(mx, dev, stream, hbm_peak: float, rows: int = 16384, K: int = 4096) -> dict:
    """The MXFP8 producer (bf16 rows -> E4M3 + 128x4-layout UE8M0 scales) on the
    largest row count the pages measure; inputs and outputs (201 MB) exceed L2."""
    import torch

    g = torch.Generator(device=dev)
    g.manual_seed(0)
    x = torch.randn((rows, K), generator=g, device=dev).to(torch.bfloat16)
    q = torch.empty((rows, K), dtype=torch.uint8, device=dev)
    sf = torch.empty(mx.moe_mxfp8_scale_bytes(rows, K, mx.MOE_SF_128X4), dtype=torch.uint8,
                     device=dev)
    times = []
    with torch.cuda.stream(stream):
        for i in range(13):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            mx.moe_mxfp8_quantize(x, rows, K, q, sf, mx.MOE_SF_128X4, rows, stream)
            b.record(stream)
            b.synchronize()
            if i >= 3:
                times.append(a.elapsed_time(b))
    alg = rows * K * 3 + sf.numel()          # bf16 read, E4M3 + scales written
    ms = statistics.mean(times)
    return {"rows": rows, "K": K, "layout": "128x4", "us": ms * 1e3,
            "achieved_GBs": alg / (ms / 1e3) / 1e9, "peak_GBs": hbm_peak,
            "frac": alg / (ms / 1e3) / 1e9 / hbm_peak, "algorithmic_bytes": alg}


def kernel_source_hash() -> str:
    with open(os.path.join(ROOT, "block_scaled_fp4_pre_gb300", "csrc", "gemm.cu"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profile_fields(text: str) -> dict:
    """The `- key: `value`` lines of a profile summary (keys may hold colons)."""
    vals = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].rsplit(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    return vals


def recorded_traffic(kernel: str, workload_name: str):
    """DRAM bytes per launch from a committed ncu summary, if it still matches gemm.cu."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_kernel_{workload_name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = profile_fields(text)
    if vals.get("gemm.cu sha256[:16]") != kernel_source_hash():
        return None
    try:
        return float(vals["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)

def oracle_sample(w: synth.Workload, x, ids, tw, n_tokens: int, nv: bool = False):
    import oracle
    from tests.helpers import compact_problem, oracle_expert_weights, oracle_expert_weights_nvf4

    tokens = np.arange(min(n_tokens, w.T))
    sub, experts = compact_problem(ids, tokens)
    # offline weight preparation, untimed
    Wc = (oracle_expert_weights_nvf4 if nv else oracle_expert_weights)(w, experts)
    return tokens, sub, Wc


def time_oracle(w, x, ids, tw, n_tokens: int, repeats: int = 1, min_seconds: float = 0.0,
                act_fp8: bool = False, nv: bool = False, nthreads: int | None = None):
    """The oracle on the first n_tokens tokens (with all their experts), run `repeats`
    times, or more until min_seconds of CPU work have been timed (at most 64 runs)."""
    import oracle

    layer = oracle.moe_w4a8 if act_fp8 else oracle.moe_nvf4 if nv else oracle.moe
    tokens, sub, Wc = oracle_sample(w, x, ids, tw, n_tokens, nv)
    times = []
    while len(times) < repeats or (sum(times) < min_seconds and len(times) < 64):
        t0 = time.perf_counter()
        layer(x[tokens], sub, tw[tokens], *Wc, nthreads=nthreads)
        times.append(time.perf_counter() - t0)
    return {"tokens": len(tokens), "seconds": times, "threads": nthreads or oracle.threads()}


def default_cpu_tokens(w):
    return 24 if w.H >= 4096 else min(w.T, 512)


# ---------------------------------------------------------------------------

def dist_setup(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    """The slowest rank's time: every replica's step must be over for the job's step."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, slowest_ms: float) -> float:
    """Whole-job throughput of `world` replicas that each process tokens_per_rank per step."""
    return world * tokens_per_rank / (slowest_ms / 1e3)


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(args)
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    n = args.cpu_sample_tokens or max(4, default_cpu_tokens(w) // 3)
    import oracle

    layer = oracle.moe_w4a8 if w4a8(args) else oracle.moe_nvf4 if nvf4(args) else oracle.moe
    tokens, sub, Wc = oracle_sample(w, x, ids, tw, n, nvf4(args))
    for _ in range(args.warmup):
        layer(x[tokens[:2]], sub[:2], tw[tokens[:2]], *Wc)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        layer(x[tokens], sub, tw[tokens], *Wc)
    dt = (time.perf_counter() - t0) / args.steps
    value = len(tokens) / dt
    line = {
        "impl": "reference", "metric": metric(args), "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(config_dict(w, world), dispatch=args.dispatch, mma_type=args.mma),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads(),
                         "kind": "oracle",
                         "sample": f"first {len(tokens)} of {w.T} tokens per step, all their experts"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(w, world):
    return {"workload": w.name, "tokens": w.T, "hidden": w.H, "inter": w.I, "experts": w.E,
            "topk": w.k, "routing": w.routing, "parallelism": f"replicas{world}",
            "l2": "flushed between timed steps (512 MiB write, then 256 MiB read so the "
                  "flush's dirty lines drain before the step); weights are 26x the L2"}


def measure_other_workload(mx, dev, stream, w: synth.Workload, prepared, args, flush_l2,
                           hbm_peak: float, fp4_peak: float, probe_best) -> dict:
    """One more layer configuration on the already prepared weights: the same step
    (pre_dispatch + forward), L2 flushed before each, CUDA events on the launch stream;
    a second pass with the library's per-kernel events gives the layer kernel's time."""
    import torch

    dims = mx.make_dims(w.H, w.I, w.E, w.k, w.T,
                        mx.MOE_MMA_FP8xFP4 if w4a8(args) else
                        mx.MOE_MMA_NVF4xNVF4 if nvf4(args) else mx.MOE_MMA_MXF4xMXF4)
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    idd = torch.from_numpy(ids).to(dev)
    twd = torch.from_numpy(tw).to(dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mx.moe_workspace_size(dims), dtype=torch.uint8, device=dev)
    mx.moe_workspace_init(dims, ws, stream)
    mx.moe_workspace_set_tiles(ws, tile_modes(mx)[args.tiles])
    mx.moe_workspace_set_dispatch(ws, mx.MOE_DISPATCH_PULL if args.dispatch == "pull"
                                  else mx.MOE_DISPATCH_BUCKETED)

    def step():
        mx.moe_pre_dispatch(dims, xd, idd, twd, w.T, ws, stream)
        mx.moe_forward(dims, prepared, ws, out, w.T, stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, min(args.warmup, 5))):
            flush_l2()
            step()
    mx.moe_check(ws, stream)
    steps = max(3, args.steps)

    def timed(profile: bool):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        mx.moe_profile_reset()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            mx.moe_profile_enable(profile)
            for i in range(steps):
                flush_l2()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            mx.moe_profile_enable(False)
        torch.cuda.synchronize(dev)
        mx.moe_check(ws, stream)
        return [a.elapsed_time(b) for a, b in zip(starts, ends)], mx.moe_profile_read()

    step_ms, _ = timed(False)
    _, per_kernel = timed(True)
    kern_ms = {k: v[0] / max(v[1], 1) for k, v in per_kernel.items()}
    ms = statistics.mean(step_ms)
    alg = algorithmic(w, ids, w4a8(args), 16 if nvf4(args) else 32)
    lay_ms = kern_ms.get("layer", float("nan"))
    achieved = alg["layer_kernel_bytes"] / (lay_ms / 1e3) / 1e9
    tflops = alg["flops"] / (lay_ms / 1e3) / 1e12
    name = w.name + ("" if args.mma == "mxf4xmxf4" else "_" + args.mma)
    traffic = recorded_traffic("layer", name)
    res = {
        "tokens": w.T, "routing": w.routing, "us_per_layer": ms * 1e3,
        "tokens_per_s": w.T / (ms / 1e3), "steps": steps,
        "step_us_min": min(step_ms) * 1e3,
        "kernels_ms": kern_ms,
        "touched_experts": alg["touched_experts"],
        "layer_kernel": {
            "avg_ms": lay_ms,
            "algorithmic_bytes": alg["layer_kernel_bytes"],
            "hbm_GBs": achieved, "hbm_frac": achieved / hbm_peak,
            "hbm_frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
            "algorithmic_flops": alg["flops"], "tflops": tflops,
            "tensor_frac": tflops / fp4_peak,
            "tensor_frac_of_mma_probe": (tflops / probe_best) if probe_best else None,
            "traffic": traffic,
            "traffic_over_algorithmic": (traffic / alg["layer_kernel_bytes"]) if traffic else None,
        },
    }
    del ws, xd, idd, twd, out
    torch.cuda.empty_cache()
    return res


def tile_modes(mx) -> dict:
    return {"auto": mx.MOE_TILES_AUTO, "wide": mx.MOE_TILES_WIDE,
            "medium": mx.MOE_TILES_MEDIUM, "narrow": mx.MOE_TILES_NARROW,
            "pair": mx.MOE_TILES_PAIR}


def run_ours(args):
    import torch

    import block_scaled_fp4_pre_gb300 as mx
    from block_scaled_fp4_pre_gb300 import weights as mxw

    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload(args)
    dims = mx.make_dims(w.H, w.I, w.E, w.k, w.T,
                        mx.MOE_MMA_FP8xFP4 if w4a8(args) else
                        mx.MOE_MMA_NVF4xNVF4 if nvf4(args) else mx.MOE_MMA_MXF4xMXF4)
    stream = torch.cuda.Stream(dev)

    t_setup = time.perf_counter()
    can = mxw.quantize_experts(dims, lambda e, o: synth.expert_w1_f32(w, e, out=o),
                               lambda e, o: synth.expert_w2_f32(w, e, out=o), dev, stream)
    prepared = mxw.prepare(dims, can, dev, stream)
    stream.synchronize()
    del can
    torch.cuda.empty_cache()
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    idd = torch.from_numpy(ids).to(dev)
    twd = torch.from_numpy(tw).to(dev)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mx.moe_workspace_size(dims), dtype=torch.uint8, device=dev)
    mx.moe_workspace_init(dims, ws, stream)
    mx.moe_workspace_set_tiles(ws, tile_modes(mx)[args.tiles])
    mx.moe_workspace_set_dispatch(ws, mx.MOE_DISPATCH_PULL if args.dispatch == "pull"
                                  else mx.MOE_DISPATCH_BUCKETED)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        clean.max()
    setup_s = time.perf_counter() - t_setup

    def step():
        mx.moe_pre_dispatch(dims, xd, idd, twd, w.T, ws, stream)
        mx.moe_forward(dims, prepared, ws, out, w.T, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            step()
    mx.moe_check(ws, stream)

    def timed_pass(profile: bool):
        """K steps, L2 flushed before each; CUDA events on the launch stream bracket
        each step.  With profile=True the library also records events around each
        of its kernels (which can keep consecutive kernels from overlapping), so the
        headline numbers come from the plain pass."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        mx.moe_profile_reset()
        barrier(world)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            mx.moe_profile_enable(profile)
            for i in range(args.steps):
                flush_l2()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            mx.moe_profile_enable(False)
        torch.cuda.synchronize(dev)
        barrier(world)
        mx.moe_check(ws, stream)
        return [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)], mx.moe_profile_read()

    def timed_graph_pass():
        """The same step captured once as a CUDA graph and replayed K times, L2
        flushed (eagerly) before each replay."""
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            step()
        with torch.cuda.stream(stream):
            for _ in range(2):
                flush_l2()
                graph.replay()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush_l2()
                starts[i].record(stream)
                graph.replay()
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        mx.moe_check(ws, stream)
        return [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]

    with ClockSampler(local) as clocks:
        step_ms, _ = timed_pass(False)
        prof_step_ms, per_kernel = timed_pass(True)
        graph_ms = timed_graph_pass()
    # the FP4 MMA probe measures kind::mxf4; it is no roof for the other MMA kinds
    probe = None if args.mma != "mxf4xmxf4" else fp4_mma_probe(mx, ws, stream,
                                                               mx.moe_device_sm_count())
    ms_local = statistics.mean(step_ms)
    ms = max_over_ranks(world, ms_local)
    value = job_tokens_per_s(world, w.T, ms)

    alg = algorithmic(w, ids, w4a8(args), 16 if nvf4(args) else 32)
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    kern_ms = {k: v[0] / max(v[1], 1) for k, v in per_kernel.items()}
    dominant = "layer"
    dom_bytes = alg["layer_kernel_bytes"]
    dom_ms = kern_ms.get(dominant, float("nan"))
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    traffic = recorded_traffic(dominant, w.name + ("" if args.mma == "mxf4xmxf4" else "_" + args.mma))
    # the tensor roof of the MMA kind: FP4 rate (mxf4) or FP8 rate (mxf8f6f4)
    ratio = FP8_PER_BF16 if w4a8(args) else FP4_PER_BF16
    fp4_peak = fp4_peak_from_bf16(peaks) * ratio / FP4_PER_BF16
    flops_achieved = alg["flops"] / (dom_ms / 1e3) / 1e12
    # The binding roof is the one that allows the longer time.
    t_hbm = dom_bytes / (hbm_peak * 1e9)
    t_fp4 = alg["flops"] / (fp4_peak * 1e12)
    hbm_roof = {"kernel": dominant, "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                "algorithmic_bytes": dom_bytes, "avg_ms": dom_ms,
                "peak_kind": f"{peak_kind} copy bandwidth"}
    tensor_roof = {"kernel": dominant, "bound": "tensor", "achieved": flops_achieved,
                   "peak": fp4_peak, "unit": "TFLOP/s", "frac": flops_achieved / fp4_peak,
                   "traffic": traffic, "algorithmic_flops": alg["flops"], "avg_ms": dom_ms,
                   "peak_kind": f"{peak_kind} bf16 GEMM burst x {ratio:g} (nominal "
                                f"{'FP8' if w4a8(args) else 'FP4'}:bf16)",
                   "mma_probe_tflops": probe}
    hbm_roof["frac_of_nominal_8tbs"] = achieved / NOMINAL_HBM_GBS
    roof, other_roof = (hbm_roof, tensor_roof) if t_hbm >= t_fp4 else (tensor_roof, hbm_roof)

    # The other DeepSeek-V4-Flash configurations, on the same prepared weights.
    workloads = None
    if not args.no_workloads and rank == 0 and args.workload == "layer_T512" and \
            not (args.experts or args.tokens):
        probe_best = max(probe.values()) if probe else None
        workloads = {}
        with ClockSampler(local) as wclocks:
            for name in OTHER_WORKLOADS:
                workloads[name] = measure_other_workload(
                    mx, dev, stream, synth.WORKLOADS[name], prepared, args, flush_l2,
                    hbm_peak, fp4_peak, probe_best)
        workloads["clocks"] = wclocks.summary()

    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(x.view(np.int16)).pin_memory()
        idh = torch.from_numpy(ids).pin_memory()
        twh = torch.from_numpy(tw).pin_memory()
        outh = torch.empty((w.T, w.H), dtype=torch.int16).pin_memory()
        for _ in range(max(1, args.warmup)):
            mx.moe_run_host(dims, prepared, ws, xh, idh, twh, outh, w.T, stream)
        times = []
        for _ in range(args.steps):
            with torch.cuda.stream(stream):
                flush_l2()
            stream.synchronize()
            t0 = time.perf_counter()
            mx.moe_run_host(dims, prepared, ws, xh, idh, twh, outh, w.T, stream)
            times.append(time.perf_counter() - t0)
        e2e_s = max_over_ranks(world, statistics.mean(times))
        e2e = {"value": job_tokens_per_s(world, w.T, e2e_s * 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": w.T * w.H * 2 + w.T * w.k * 8,
               "d2h_bytes_per_step": w.T * w.H * 2, "ms_per_step": e2e_s * 1e3}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = args.cpu_sample_tokens or default_cpu_tokens(w)
        r = time_oracle(w, x, ids, tw, n, min_seconds=10.0, act_fp8=w4a8(args), nv=nvf4(args))
        runs, secs = len(r["seconds"]), sum(r["seconds"])
        cpu = {"value": r["tokens"] * runs / secs, "unit": "tokens/s", "cores": r["threads"],
               "kind": "oracle",
               "sample": f"first {r['tokens']} of {w.T} tokens with all {w.k} experts each, "
                         f"{runs} runs ({secs:.1f} s of oracle time)"}
        # the same oracle on one thread, on a third of the sample
        r1 = time_oracle(w, x, ids, tw, max(2, n // 3), min_seconds=5.0, act_fp8=w4a8(args),
                         nv=nvf4(args), nthreads=1)
        runs1, secs1 = len(r1["seconds"]), sum(r1["seconds"])
        cpu["single_thread"] = {"value": r1["tokens"] * runs1 / secs1, "unit": "tokens/s",
                                "cores": 1,
                                "sample": f"first {r1['tokens']} tokens, {runs1} runs "
                                          f"({secs1:.1f} s)"}

    if rank != 0:
        return
    vs, vs_basis = pages_ratio(args, w, world, value)
    line = {
        "metric": metric(args),
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "us_per_layer": ms * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": vs,
        "vs_baseline_basis": vs_basis,
        "dtype": ("mxfp4 weights (e2m1 x ue8m0) x mxfp8 activations (e4m3 x ue8m0), fp32 accumulate"
                  if w4a8(args) else
                  "nvfp4 (e2m1 x ue4m3 per 16), fp32 accumulate" if nvf4(args) else
                  "mxfp4 (e2m1 x ue8m0), fp32 accumulate"),
        "data": "synthetic",
        "config": dict(config_dict(w, world), dispatch=args.dispatch, mma_type=args.mma,
                       tiles=args.tiles),
        "layer_hbm_tbs": alg["layer_bytes"] / (ms / 1e3) / 1e12,
        "layer_roofline_frac": (alg["layer_bytes"] / (hbm_peak * 1e9)) / (ms / 1e3),
        "touched_experts": alg["touched_experts"],
        "roofline": roof,
        "roofline_other": other_roof,
        "kernels_ms": kern_ms,
        "step_us": {"mean": ms_local * 1e3, "median": statistics.median(step_ms) * 1e3,
                    "min": min(step_ms) * 1e3},
        "graph_step_us": {"mean": statistics.mean(graph_ms) * 1e3,
                          "median": statistics.median(graph_ms) * 1e3,
                          "min": min(graph_ms) * 1e3},
        "profiled_ms_per_step": statistics.mean(prof_step_ms),
        "mxfp8_producer": mxfp8_producer(mx, dev, stream, hbm_peak),
        "clocks": clocks.summary(),
        "gpu_launches": KERNELS_PER_STEP * args.steps,   # in the headline timed pass
        "setup_s": setup_s,
    }
    if workloads is not None:
        line["workloads"] = workloads
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

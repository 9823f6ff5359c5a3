"""CUDA path against the CPU oracle, through the C ABI (GB300 only).

Bars: quantised codes, scales and bucketing bit-exact; gate/up accumulators within
fp32 accumulation error of the exact sums; intermediate FP4 codes differing in at
most 0.1% of elements, each by one grid step; final output normwise relative error
<= 2e-3 against the oracle (before its bf16 rounding and after it).
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_scaled_fp4_pre_gb300 as mx  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from tests.gpu_common import (DeviceLayer, compare_full, device, full_size_check,  # noqa: E402
                              to_dev)
from tests.helpers import (normwise_rel_err, oracle_expert_weights,  # noqa: E402
                           untile_codes)

pytestmark = pytest.mark.gpu

# Small shapes that span several tiles, ragged token tails and a ragged K block.
SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    # ~175 tokens per expert: two token tiles each (128 + tail); I = 384 gives a
    # 128-wide last k-block in the down projection; 6 gate/up slabs, 4 down slabs.
    "ragged": synth.Workload("ragged", T=700, H=512, I=384, E=8, k=2),
    # skewed routing: expert 0 gets several tiles, the rarest a handful of tokens
    "zipf": synth.Workload("zipf", T=1024, H=256, I=256, E=32, k=4, routing="zipf",
                           outlier_frac=0.001),
    "top1": synth.Workload("top1", T=96, H=256, I=128, E=1, k=1),
    # 256 rows per expert (wide tiles) with an odd number of down slabs (H/128 = 3),
    # so block pairs stay off, and a 128-wide last k-block in the gate/up phase
    "oddslab": synth.Workload("oddslab", T=512, H=384, I=256, E=4, k=2),
}


@pytest.fixture(scope="module")
def layers():
    cache = {}

    def get(name):
        if name not in cache:
            w = SMALL[name]
            cache[name] = (DeviceLayer(w, keep_canonical=True), oracle_expert_weights(w, range(w.E)))
        return cache[name]

    return get


# --------------------------------------------------------------------------
# Quantiser

def test_quantize_mxfp4_bit_exact_adversarial():
    rng = np.random.default_rng(11)
    rows = [rng.standard_normal(256) * 10.0 ** rng.uniform(-6, 6) for _ in range(64)]
    ties = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 32)
    rows += [ties, -ties, ties * 2.0 ** -100, ties * 2.0 ** 100]
    z = np.zeros(256); z[5] = -0.0; z[9] = -1e-40; rows.append(z)
    rows.append(np.full(256, 6.0 * (1 + 2.0 ** -23)))
    rows.append(np.full(256, 2.0 ** -130))
    o = rng.standard_normal(256); o[::37] *= 50; rows.append(o)
    x = np.stack(rows).astype(np.float32)
    codes = torch.empty((x.shape[0], 128), dtype=torch.uint8, device=device())
    sf = torch.empty((x.shape[0], 8), dtype=torch.uint8, device=device())
    mx.moe_quantize_mxfp4(to_dev(x), codes, sf)
    rc, rs = oracle.quantize_f32(x)
    assert np.array_equal(sf.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantize_mxfp4_all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32)
    finite = (bits & 0x7F80) != 0x7F80
    vals = ((bits[finite] << 16).astype(np.uint32)).view(np.float32)
    rng = np.random.default_rng(12)
    vals = vals[rng.permutation(vals.size)]            # mix magnitudes inside groups
    pad = (-vals.size) % 256
    vals = np.concatenate([vals, np.zeros(pad, np.float32)]).reshape(-1, 256)
    sorted_vals = np.sort(np.abs(vals.reshape(-1))).reshape(-1, 256)   # and similar ones together
    x = np.concatenate([vals, sorted_vals]).astype(np.float32)
    codes = torch.empty((x.shape[0], 128), dtype=torch.uint8, device=device())
    sf = torch.empty((x.shape[0], 8), dtype=torch.uint8, device=device())
    mx.moe_quantize_mxfp4(to_dev(x), codes, sf)
    rc, rs = oracle.quantize_f32(x)
    assert np.array_equal(sf.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


# --------------------------------------------------------------------------
# Weight preparation

@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_weights_quantised_and_prepared_bit_exact(layers, name):
    layer, W = layers(name)
    w = layer.w
    can = {k: v.cpu().numpy() for k, v in layer.canonical.items()}
    for got, ref in zip((can["w1_codes"], can["w1_scales"], can["w2_codes"], can["w2_scales"]), W):
        assert np.array_equal(got, ref)
    blob = layer.prepared.cpu().numpy()
    src = oracle.interleave_source_rows(w.I)
    E, H, I = w.E, w.H, w.I
    w1c_p = W[0][:, src, :]
    w1s_p = W[1][:, src, :]
    off = 0
    n = E * 2 * I * -(-H // 256) * 128
    assert np.array_equal(untile_codes(blob[off:off + n], E * 2 * I, H), w1c_p.reshape(E * 2 * I, -1))
    off = (off + n + 1023) // 1024 * 1024
    n = E * 2 * I * H // 32
    assert np.array_equal(blob[off:off + n], oracle.scale_block_layout(w1s_p.reshape(E * 2 * I, -1)))
    off = (off + n + 1023) // 1024 * 1024
    n = E * H * -(-I // 256) * 128
    assert np.array_equal(untile_codes(blob[off:off + n], E * H, I), W[2].reshape(E * H, -1))
    off = (off + n + 1023) // 1024 * 1024
    n = E * H * I // 32
    assert np.array_equal(blob[off:off + n], oracle.scale_block_layout(W[3].reshape(E * H, -1)))


# --------------------------------------------------------------------------
# pre_dispatch

@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf", "top1"])
def test_pre_dispatch_bit_exact(layers, name):
    layer, W = layers(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w) if w.E > 1 else (np.zeros((w.T, 1), np.int32),
                                                 np.ones((w.T, 1), np.float32))
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    mx.moe_check(layer.ws)
    d = mx.moe_read_dispatch(layer.dims, layer.ws, w.T)
    counts, offsets, st, sj, bad = oracle.bucket(ids, w.E)
    assert bad == 0
    assert np.array_equal(d["counts"], counts)
    assert np.array_equal(d["slot_token"], np.repeat(np.arange(w.T), w.k))
    # within an expert the rows follow ascending (t, j): the oracle's slot order
    slot = d["assign_slot"]
    for e in range(w.E):
        a_sorted = (st[offsets[e]:offsets[e + 1]].astype(np.int64) * w.k + sj[offsets[e]:offsets[e + 1]])
        rows = slot[a_sorted]
        assert np.all(np.diff(rows) == 1)
    xc, xs = oracle.quantize_bf16(x)
    assert np.array_equal(d["x_codes"], np.repeat(xc, w.k, axis=0))
    assert np.array_equal(d["x_scales"], np.repeat(xs, w.k, axis=0))


# --------------------------------------------------------------------------
# Gate/up GEMM accumulators

@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf"])
def test_gate_up_accumulators(layers, name):
    layer, W = layers(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    gu = torch.full((w.T * w.k, 2 * w.I), float("nan"), dtype=torch.float32, device=device())
    mx.moe_debug_gate_up(layer.dims, layer.prepared, layer.ws, gu, w.T)
    mx.moe_check(layer.ws)
    got = gu.cpu().numpy().astype(np.float64)
    ref = oracle.moe(x, ids, tw, *W, want_intermediates=True)["gate_up"]
    xd = np.abs(oracle.dequantize(*oracle.quantize_bf16(x)))
    wd = [np.abs(oracle.dequantize(W[0][e], W[1][e])) for e in range(w.E)]
    bound = np.zeros_like(ref)
    for t in range(w.T):
        for j in range(w.k):
            bound[t * w.k + j] = wd[ids[t, j]] @ xd[t]
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= 1e-5 * bound + 1e-30)


# --------------------------------------------------------------------------
# Whole layer

@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf", "top1", "oddslab"])
def test_forward_matches_oracle(layers, name):
    layer, W = layers(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w) if w.E > 1 else (np.zeros((w.T, 1), np.int32),
                                                 np.ones((w.T, 1), np.float32))
    got = layer.run(x, ids, tw)
    m = compare_full(layer, x, ids, tw, got, W)
    print(name, {k: v for k, v in m.items() if k != "ref"})
    assert m["flip_frac"] <= 1e-3 and m["flips_one_step"]
    assert m["err_f64"] <= 2e-3
    assert m["err_bf16"] <= 2e-3
    # down projection + combine alone, on the GPU's own intermediate codes
    assert m["err_own_h"] <= 2e-3 and m["own_h_bf16_equal"] >= 0.99


def test_forward_is_repeatable_and_host_path_matches(layers):
    layer, W = layers("ragged")
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    a = layer.run(x, ids, tw)
    inter_a = mx.moe_read_intermediate(layer.dims, layer.ws, w.T)
    b = layer.run(x, ids, tw)
    inter_b = mx.moe_read_intermediate(layer.dims, layer.ws, w.T)
    assert np.array_equal(inter_a["h_codes"], inter_b["h_codes"])
    # fp32 reductions in arbitrary order: outputs agree to bf16 rounding
    assert normwise_rel_err(oracle.bf16_bits_to_f64(a), oracle.bf16_bits_to_f64(b)) <= 1e-3
    # page-locked buffers are accessed in place, pageable ones staged; all and none
    # page-locked, then a mix
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    idh, twh = torch.from_numpy(ids).pin_memory(), torch.from_numpy(tw).pin_memory()
    for args in [(xh, idh, twh, torch.empty((w.T, w.H), dtype=torch.int16).pin_memory()),
                 (np.ascontiguousarray(x.view(np.int16)), ids, tw, np.zeros((w.T, w.H), np.int16)),
                 (np.ascontiguousarray(x.view(np.int16)), idh, tw, torch.zeros((w.T, w.H), dtype=torch.int16).pin_memory()),
                 (xh, ids, twh, np.zeros((w.T, w.H), np.int16))]:
        mx.moe_run_host(layer.dims, layer.prepared, layer.ws, *args, w.T)
        c = np.asarray(args[3]).view(np.uint16)
        assert normwise_rel_err(oracle.bf16_bits_to_f64(c), oracle.bf16_bits_to_f64(a)) <= 1e-3


def test_cuda_graph_replay_matches_eager(layers):
    """pre_dispatch + forward captured as one CUDA graph (the calls neither
    synchronise nor allocate) and replayed: same intermediate codes as an eager run,
    same output up to the order of the fp32 reductions."""
    layer, W = layers("zipf")
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    eager = layer.run(x, ids, tw)
    inter_e = mx.moe_read_intermediate(layer.dims, layer.ws, w.T)
    xd, idd, twd = to_dev(x), to_dev(ids), to_dev(tw)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=device())
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        mx.moe_pre_dispatch(layer.dims, xd, idd, twd, w.T, layer.ws, s)
        mx.moe_forward(layer.dims, layer.prepared, layer.ws, out, w.T, s)
    for _ in range(3):
        out.fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        mx.moe_check(layer.ws, s)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert normwise_rel_err(oracle.bf16_bits_to_f64(got), oracle.bf16_bits_to_f64(eager)) <= 1e-3
    inter_g = mx.moe_read_intermediate(layer.dims, layer.ws, w.T)
    assert np.array_equal(inter_g["h_codes"], inter_e["h_codes"])
    assert np.array_equal(inter_g["h_scales"], inter_e["h_scales"])


def test_forward_twice_on_one_pre_dispatch(layers):
    layer, W = layers("ragged")
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=device())
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    mx.moe_forward(layer.dims, layer.prepared, layer.ws, out, w.T)
    first = out.view(torch.int16).cpu().numpy().view(np.uint16)
    out.zero_()
    mx.moe_forward(layer.dims, layer.prepared, layer.ws, out, w.T)   # no new pre_dispatch
    mx.moe_check(layer.ws)
    second = out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.moe(x, ids, tw, *W)
    for got in (first, second):
        assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3


def test_partial_batch_and_edge_token_counts(layers):
    layer, W = layers("ragged")
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    for T in (1, 2, 127, 129):
        got = layer.run(x[:T], ids[:T], tw[:T])
        ref = oracle.moe(x[:T], ids[:T], tw[:T], *W)
        assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3, T
    # zero tokens is a no-op
    out = torch.empty((1, w.H), dtype=torch.bfloat16, device=device())
    mx.moe_pre_dispatch(layer.dims, out, out, out, 0, layer.ws)
    mx.moe_forward(layer.dims, layer.prepared, layer.ws, out, 0)


def test_all_tokens_on_one_expert(layers):
    layer, W = layers("ragged")
    w = layer.w
    T = w.T
    x = synth.hidden_bf16(w)
    ids = np.stack([np.full(T, 3), np.full(T, 5)], axis=1).astype(np.int32)   # 700 rows each
    tw = np.full((T, 2), 0.5, np.float32)
    got = layer.run(x, ids, tw)
    ref = oracle.moe(x, ids, tw, *W)
    assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3


def test_invalid_ids_are_skipped_and_reported(layers):
    layer, W = layers("tiny")
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    bad = ids.copy()
    bad[2, 0] = -1
    bad[7, 1] = w.E
    T = w.T
    out = torch.empty((T, w.H), dtype=torch.bfloat16, device=device())
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(bad), to_dev(tw), T, layer.ws)
    mx.moe_forward(layer.dims, layer.prepared, layer.ws, out, T)
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_check(layer.ws)
    assert ei.value.status == mx.MOE_ERR_ROUTING
    mx.moe_check(layer.ws)          # the flag was cleared
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.moe(x, bad, tw, *W)
    assert ref["invalid_ids"] == 2
    assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3


def test_bounded_wait_reports_timeout_and_context_survives(layers):
    layer, W = layers("tiny")
    w = layer.w
    mx.moe_check(layer.ws)
    mx.moe_debug_wait_probe(layer.ws, 10_000_000)       # 10 ms per wait
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_check(layer.ws)
    assert ei.value.status == mx.MOE_ERR_TIMEOUT
    mx.moe_check(layer.ws)                              # reported once, then cleared
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    got = layer.run(x, ids, tw)                         # the context still works
    ref = oracle.moe(x, ids, tw, *W)
    assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3


def test_fp4_mma_probe_runs_and_rejects_bad_shapes(layers):
    """The FP4 throughput probe completes with a clean status at each tile shape, and
    its rate is plausible for the part: below the nominal dense FP4 peak with margin
    (13.5 PFLOP/s; a rate above it would mean the timed launch skipped work) and
    above a tenth of it."""
    layer, _ = layers("tiny")
    sms = mx.moe_device_sm_count()
    for n, bps in ((32, 2), (128, 2), (256, 1)):
        count = 1 << 16
        mx.moe_fp4_mma_probe(layer.ws, n, bps, sms * bps, count)    # warm-up
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        mx.moe_fp4_mma_probe(layer.ws, n, bps, sms * bps, count)
        b.record()
        b.synchronize()
        mx.moe_check(layer.ws)
        tflops = sms * bps * count * 2.0 * 128 * n * 64 / (a.elapsed_time(b) / 1e3) / 1e12
        if n >= 128:
            assert 1350 < tflops < 1.2 * 13500, (n, bps, tflops)
    for bad in ((48, 2, sms, 16), (256, 2, sms, 16), (128, 3, sms, 16), (128, 2, 0, 16),
                (128, 2, sms, 0), (128, 2, sms, (1 << 20) + 1)):
        with pytest.raises(mx.MoeError) as ei:
            mx.moe_fp4_mma_probe(layer.ws, *bad)
        assert ei.value.status == mx.MOE_ERR_INVALID_ARG
    # the M=256 form across SM pairs (tcgen05 cta_group::2)
    pairs, count = sms // 2, 1 << 16
    for n in (128, 256):
        mx.moe_fp4_mma_probe_pair(layer.ws, n, pairs, count)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        mx.moe_fp4_mma_probe_pair(layer.ws, n, pairs, count)
        b.record()
        b.synchronize()
        mx.moe_check(layer.ws)
        tflops = pairs * count * 2.0 * 256 * n * 64 / (a.elapsed_time(b) / 1e3) / 1e12
        assert 1350 < tflops < 1.2 * 13500, (n, tflops)
    for bad in ((48, pairs, 16), (288, pairs, 16), (128, 0, 16), (128, pairs, 0)):
        with pytest.raises(mx.MoeError) as ei:
            mx.moe_fp4_mma_probe_pair(layer.ws, *bad)
        assert ei.value.status == mx.MOE_ERR_INVALID_ARG


def test_workspace_checks(layers):
    layer, _ = layers("tiny")
    other = mx.make_dims(layer.dims.hidden, layer.dims.inter, layer.dims.num_experts,
                         layer.dims.topk, layer.dims.max_tokens + 1)
    x = torch.zeros((1, layer.dims.hidden), dtype=torch.bfloat16, device=device())
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_pre_dispatch(other, x, x, x, 1, layer.ws)
    assert ei.value.status in (mx.MOE_ERR_WORKSPACE_MISMATCH, mx.MOE_ERR_WORKSPACE_TOO_SMALL)
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_pre_dispatch(layer.dims, x, x, x, layer.dims.max_tokens + 1, layer.ws)
    assert ei.value.status == mx.MOE_ERR_INVALID_ARG


# --------------------------------------------------------------------------
# Full DeepSeek-V4-Flash shape, in the launch configuration the benchmark times:
# every expert on the device, outputs of sampled tokens against the oracle.

@pytest.fixture(scope="module")
def dsv4_layer():
    w = synth.WORKLOADS["prefill_T16384_zipf"]
    return DeviceLayer(w, max_tokens=w.T)


@pytest.fixture(scope="module")
def dsv4_weight_cache():
    """Oracle-side weights by expert, shared by the DeepSeek-V4-Flash configurations
    (they have the same H, I and E)."""
    return {}


@pytest.mark.parametrize("name", ["decode_T64", "layer_T512", "prefill_T4096",
                                  "prefill_T16384_zipf"])
def test_full_size_against_oracle(dsv4_layer, dsv4_weight_cache, name):
    """Every DeepSeek-V4-Flash configuration at full size: bucketing and every token
    row bit-exact; intermediate flips within 0.1% (one step each) and outputs within
    2e-3 normwise on the checked tokens -- all 512 tokens (3072 assignments) at T=512,
    sixteen sampled tokens (and, under skewed routing, one on the busiest expert)
    elsewhere."""
    w = synth.WORKLOADS[name]
    tokens = np.arange(w.T) if name == "layer_T512" else None
    full_size_check(dsv4_layer, w, "mxf4", tokens=tokens, weight_cache=dsv4_weight_cache)

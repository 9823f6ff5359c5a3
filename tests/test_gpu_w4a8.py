"""The fp8xfp4 (W4A8) layer on the GPU against the oracle.

Digest of SGLang PR #37279, items 1-4: mma_type "fp8xfp4" quantises the hidden
states to FP8 with quant_group_size=32 and interleaves the first weight's gate/up rows
with gran=8; the weights stay MXFP4.  The E4M3 token codes, their scales and the
bucketing must be bit-exact; the gate/up accumulators within fp32 accumulation error
of the exact sums; the intermediate's E4M3 codes may differ from the oracle's in at
most 0.1% of elements, each by one grid step; the output within 2e-3 normwise.
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
from tests.gpu_common import DeviceLayer, device, full_size_check, to_dev  # noqa: E402
from tests.gpu_common import flip_stats8  # noqa: E402
from tests.helpers import normwise_rel_err, oracle_expert_weights  # noqa: E402

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "ragged": synth.Workload("ragged", T=700, H=512, I=384, E=8, k=2),
    "zipf": synth.Workload("zipf", T=1024, H=256, I=256, E=32, k=4, routing="zipf",
                           outlier_frac=0.001),
    "oddslab": synth.Workload("oddslab", T=512, H=384, I=256, E=4, k=2),
}
_cache = {}


def _layer(name):
    if name not in _cache:
        w = SMALL[name]
        _cache[name] = (DeviceLayer(w, mma_type=mx.MOE_MMA_FP8xFP4),
                        oracle_expert_weights(w, range(w.E)))
    return _cache[name]


@pytest.mark.parametrize("name", list(SMALL))
def test_w4a8_pre_dispatch_bit_exact(name):
    layer, _ = _layer(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    mx.moe_check(layer.ws)
    d = mx.moe_read_dispatch(layer.dims, layer.ws, w.T)
    counts, _, _, _, bad = oracle.bucket(ids, w.E)
    assert bad == 0 and np.array_equal(d["counts"], counts)
    assert np.array_equal(d["slot_token"], np.repeat(np.arange(w.T), w.k))
    xq, xs = oracle.mxfp8_quantize_bf16(x)
    assert d["x_codes"].shape == (w.T * w.k, w.H)
    assert np.array_equal(d["x_codes"], np.repeat(xq, w.k, axis=0))
    assert np.array_equal(d["x_scales"], np.repeat(xs, w.k, axis=0))


@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf"])
def test_w4a8_gate_up_accumulators(name):
    layer, W = _layer(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    gu = torch.full((w.T * w.k, 2 * w.I), float("nan"), dtype=torch.float32, device=device())
    mx.moe_debug_gate_up(layer.dims, layer.prepared, layer.ws, gu, w.T)
    mx.moe_check(layer.ws)
    got = gu.cpu().numpy().astype(np.float64)
    ref = oracle.moe_w4a8(x, ids, tw, *W, want_intermediates=True)["gate_up"]
    xd = np.abs(oracle.mxfp8_dequantize(*oracle.mxfp8_quantize_bf16(x)))
    wd = [np.abs(oracle.dequantize(W[0][e], W[1][e])) for e in range(w.E)]
    bound = np.zeros_like(ref)
    for t in range(w.T):
        for j in range(w.k):
            bound[t * w.k + j] = wd[ids[t, j]] @ xd[t]
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= 1e-5 * bound + 1e-30)


@pytest.mark.parametrize("name", list(SMALL))
def test_w4a8_forward_matches_oracle(name):
    layer, W = _layer(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    got = layer.run(x, ids, tw)
    ref = oracle.moe_w4a8(x, ids, tw, *W, want_intermediates=True)
    inter = mx.moe_read_intermediate(layer.dims, layer.ws, w.T)
    assert inter["h_codes"].shape == (w.T * w.k, w.I)
    frac, one_step = flip_stats8(inter["h_codes"], inter["h_scales"], ref["h_codes"], ref["h_sf"])
    g = oracle.bf16_bits_to_f64(got)
    err = normwise_rel_err(g, ref["out_f64"])
    down = oracle.moe_w4a8_down(ids, tw, W[2], W[3], inter["h_codes"], inter["h_scales"], w.H)
    err_own = normwise_rel_err(g, down["out_f64"])
    print(name, "flips", frac, "err", err, "err_own_h", err_own)
    assert frac <= 1e-3 and one_step
    assert err <= 2e-3 and err_own <= 2e-3


def test_w4a8_pull_dispatch_is_rejected():
    layer, _ = _layer("tiny")
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_workspace_set_dispatch(layer.ws, mx.MOE_DISPATCH_PULL)
    assert ei.value.status == mx.MOE_ERR_UNSUPPORTED
    mx.moe_workspace_set_dispatch(layer.ws, mx.MOE_DISPATCH_BUCKETED)


@pytest.fixture(scope="module")
def dsv4_w4a8():
    w = synth.WORKLOADS["prefill_T16384_zipf"]
    return DeviceLayer(w, max_tokens=w.T, mma_type=mx.MOE_MMA_FP8xFP4)


@pytest.mark.parametrize("name", ["decode_T64", "layer_T512", "prefill_T4096",
                                  "prefill_T16384_zipf"])
def test_w4a8_full_size_sampled_tokens(dsv4_w4a8, name):
    """DeepSeek-V4-Flash shape in the benchmark's launch configuration: bucketing and
    every token row bit-exact; on sampled tokens, intermediate flips within 0.1% (one
    step each) and outputs within the oracle's bar."""
    full_size_check(dsv4_w4a8, synth.WORKLOADS[name], "w4a8", n_sample=8, seed=23)


@pytest.mark.parametrize("name", ["ragged", "oddslab"])
def test_w4a8_tile_widths_agree(name):
    """E4M3 tokens on 32- and 64-row tiles stage two 128-element k-blocks at a time;
    128-row tiles one.  Shapes with an odd number of k-blocks (K = 384: the last stage
    holds one) must give the same gate/up accumulators and intermediate codes on every
    tile width (the tile width changes which token rows share an MMA, not any element's
    K reduction), and outputs equal up to the order of the combine's fp32 additions."""
    layer, W = _layer(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    ref = oracle.moe_w4a8(x, ids, tw, *W)
    seen = {}
    try:
        for tiles in (mx.MOE_TILES_NARROW, mx.MOE_TILES_MEDIUM, mx.MOE_TILES_WIDE):
            mx.moe_workspace_set_tiles(layer.ws, tiles)
            mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
            gu = torch.full((w.T * w.k, 2 * w.I), float("nan"), dtype=torch.float32,
                            device=device())
            mx.moe_debug_gate_up(layer.dims, layer.prepared, layer.ws, gu, w.T)
            mx.moe_check(layer.ws)
            out = layer.run(x, ids, tw)
            inter = mx.moe_read_intermediate(layer.dims, layer.ws, w.T)
            seen[tiles] = (gu.cpu().numpy(), inter["h_codes"], inter["h_scales"], out)
            assert normwise_rel_err(oracle.bf16_bits_to_f64(out), ref["out_f64"]) <= 2e-3
    finally:
        mx.moe_workspace_set_tiles(layer.ws, mx.MOE_TILES_AUTO)
    g0, c0, s0, o0 = seen[mx.MOE_TILES_WIDE]
    assert np.all(np.isfinite(g0))
    for tiles in (mx.MOE_TILES_NARROW, mx.MOE_TILES_MEDIUM):
        g, c, sc, o = seen[tiles]
        assert np.array_equal(g, g0), tiles
        assert np.array_equal(c, c0) and np.array_equal(sc, s0), tiles
        assert normwise_rel_err(oracle.bf16_bits_to_f64(o), oracle.bf16_bits_to_f64(o0)) <= 1e-3

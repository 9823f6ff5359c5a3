"""The NVFP4 layer (nvf4xnvf4) on the GPU against the oracle.

NVFP4 here: packed E2M1 with one E4M3 scale per 16 elements (the E4M3 value nearest
to amax/6; elements fp32(x / scale) rounded to E2M1), for the weights, the tokens and
the requantised intermediate; gran=16 gate/up rows.  Weight and token codes, their
scales and the bucketing must be bit-exact; the gate/up accumulators within fp32
accumulation error of the exact sums; intermediate codes may differ from the oracle's
in at most 0.1% of elements, each by one grid step; the output within 2e-3 normwise.
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
from tests.gpu_common import flip_stats_nv  # noqa: E402
from tests.helpers import normwise_rel_err, oracle_expert_weights_nvf4  # noqa: E402

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
        _cache[name] = (DeviceLayer(w, mma_type=mx.MOE_MMA_NVF4xNVF4, keep_canonical=True),
                        oracle_expert_weights_nvf4(w, range(w.E)))
    return _cache[name]


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_nvf4_weight_quantiser_bit_exact(name):
    layer, W = _layer(name)
    can = layer.canonical
    for key, i in (("w1_codes", 0), ("w1_scales", 1), ("w2_codes", 2), ("w2_scales", 3)):
        assert np.array_equal(can[key].cpu().numpy(), W[i]), key


@pytest.mark.parametrize("name", list(SMALL))
def test_nvf4_pre_dispatch_bit_exact(name):
    layer, _ = _layer(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    mx.moe_check(layer.ws)
    d = mx.moe_read_dispatch(layer.dims, layer.ws, w.T)
    counts, _, _, _, bad = oracle.bucket(ids, w.E)
    assert bad == 0 and np.array_equal(d["counts"], counts)
    xc, xs = oracle.nvfp4_quantize_bf16(x)
    assert d["x_scales"].shape == (w.T * w.k, w.H // 16)
    assert np.array_equal(d["x_codes"], np.repeat(xc, w.k, axis=0))
    assert np.array_equal(d["x_scales"], np.repeat(xs, w.k, axis=0))


@pytest.mark.parametrize("name", ["tiny", "ragged", "zipf"])
def test_nvf4_gate_up_accumulators(name):
    layer, W = _layer(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    gu = torch.full((w.T * w.k, 2 * w.I), float("nan"), dtype=torch.float32, device=device())
    mx.moe_debug_gate_up(layer.dims, layer.prepared, layer.ws, gu, w.T)
    mx.moe_check(layer.ws)
    got = gu.cpu().numpy().astype(np.float64)
    ref = oracle.moe_nvf4(x, ids, tw, *W, want_intermediates=True)["gate_up"]
    xd = np.abs(oracle.nvfp4_dequantize(*oracle.nvfp4_quantize_bf16(x)))
    wd = [np.abs(oracle.nvfp4_dequantize(W[0][e], W[1][e])) for e in range(w.E)]
    bound = np.zeros_like(ref)
    for t in range(w.T):
        for j in range(w.k):
            bound[t * w.k + j] = wd[ids[t, j]] @ xd[t]
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= 1e-5 * bound + 1e-30)


@pytest.mark.parametrize("name", list(SMALL))
def test_nvf4_forward_matches_oracle(name):
    layer, W = _layer(name)
    w = layer.w
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    got = layer.run(x, ids, tw)
    ref = oracle.moe_nvf4(x, ids, tw, *W, want_intermediates=True)
    inter = mx.moe_read_intermediate(layer.dims, layer.ws, w.T)
    frac, one_step = flip_stats_nv(inter["h_codes"], inter["h_scales"], ref["h_codes"], ref["h_sf"])
    err = normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"])
    print(name, "flips", frac, "err", err)
    assert frac <= 1e-3 and one_step
    assert err <= 2e-3


def test_nvf4_pull_dispatch_is_rejected():
    layer, _ = _layer("tiny")
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_workspace_set_dispatch(layer.ws, mx.MOE_DISPATCH_PULL)
    assert ei.value.status == mx.MOE_ERR_UNSUPPORTED


@pytest.fixture(scope="module")
def dsv4_nvf4():
    w = synth.WORKLOADS["prefill_T16384_zipf"]
    return DeviceLayer(w, max_tokens=w.T, mma_type=mx.MOE_MMA_NVF4xNVF4)


@pytest.mark.parametrize("name", ["decode_T64", "layer_T512", "prefill_T4096",
                                  "prefill_T16384_zipf"])
def test_nvf4_full_size_sampled_tokens(dsv4_nvf4, name):
    """DeepSeek-V4-Flash shape in the benchmark's launch configuration: bucketing and
    every token row bit-exact; on sampled tokens, intermediate flips within 0.1% (one
    step each) and outputs within the oracle's bar."""
    full_size_check(dsv4_nvf4, synth.WORKLOADS[name], "nvf4", n_sample=8, seed=23)

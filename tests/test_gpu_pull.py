"""Pull dispatch (MOE_DISPATCH_PULL) against the bucketed dispatch and the oracle.

SGLang PR #48424, Summary ("SIMT dispatch pull for FP4 activations"): the layer
gathers each expert's token rows itself, from one quantised row per token, instead of
reading copies that pre_dispatch bucketed per expert.  The MMAs see the same bytes in
the same order, so the intermediate codes must be bit-identical to the bucketed
path's, the output equal up to the order of the fp32 reductions, and both within the
oracle's bars.
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
from tests.gpu_common import DeviceLayer, compare_full  # noqa: E402
from tests.helpers import compact_problem, normwise_rel_err, oracle_expert_weights  # noqa: E402

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "ragged": synth.Workload("ragged", T=700, H=512, I=384, E=8, k=2),
    "zipf": synth.Workload("zipf", T=1024, H=256, I=256, E=32, k=4, routing="zipf",
                           outlier_frac=0.001),
    # a 128-wide last k-block in the gathered gate/up phase (H % 256 == 128), and an
    # odd number of down slabs (no block pairs)
    "oddslab": synth.Workload("oddslab", T=512, H=384, I=256, E=4, k=2),
}


def _both_modes(layer, x, ids, tw):
    out = {}
    for mode in (mx.MOE_DISPATCH_BUCKETED, mx.MOE_DISPATCH_PULL):
        mx.moe_workspace_set_dispatch(layer.ws, mode)
        got = layer.run(x, ids, tw)
        inter = mx.moe_read_intermediate(layer.dims, layer.ws, x.shape[0])
        out[mode] = (got, inter, mx.moe_read_dispatch(layer.dims, layer.ws, x.shape[0]))
    return out


@pytest.mark.parametrize("name", list(SMALL))
def test_pull_matches_bucketed_and_oracle(name):
    w = SMALL[name]
    layer = DeviceLayer(w)
    W = oracle_expert_weights(w, range(w.E))
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    res = _both_modes(layer, x, ids, tw)
    got_b, inter_b, _ = res[mx.MOE_DISPATCH_BUCKETED]
    got_p, inter_p, disp_p = res[mx.MOE_DISPATCH_PULL]
    assert np.array_equal(inter_p["h_codes"], inter_b["h_codes"])
    assert np.array_equal(inter_p["h_scales"], inter_b["h_scales"])
    assert normwise_rel_err(oracle.bf16_bits_to_f64(got_p), oracle.bf16_bits_to_f64(got_b)) <= 1e-3
    xc, xs = oracle.quantize_bf16(x)
    assert np.array_equal(disp_p["x_codes"], np.repeat(xc, w.k, axis=0))
    assert np.array_equal(disp_p["x_scales"], np.repeat(xs, w.k, axis=0))
    m = compare_full(layer, x, ids, tw, got_p, W)     # the workspace holds the pull run
    assert m["flip_frac"] <= 1e-3 and m["flips_one_step"]
    assert m["err_f64"] <= 2e-3 and m["err_bf16"] <= 2e-3


def test_pull_gate_up_accumulators_equal_bucketed():
    w = SMALL["ragged"]
    layer = DeviceLayer(w)
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    acc = {}
    for mode in (mx.MOE_DISPATCH_BUCKETED, mx.MOE_DISPATCH_PULL):
        mx.moe_workspace_set_dispatch(layer.ws, mode)
        mx.moe_pre_dispatch(layer.dims, torch.from_numpy(x.view(np.int16)).cuda(),
                            torch.from_numpy(ids).cuda(), torch.from_numpy(tw).cuda(), w.T, layer.ws)
        gu = torch.full((w.T * w.k, 2 * w.I), float("nan"), dtype=torch.float32, device="cuda")
        mx.moe_debug_gate_up(layer.dims, layer.prepared, layer.ws, gu, w.T)
        mx.moe_check(layer.ws)
        acc[mode] = gu.cpu().numpy()
    assert np.array_equal(acc[mx.MOE_DISPATCH_PULL], acc[mx.MOE_DISPATCH_BUCKETED])


def test_dispatch_mode_argument_checks():
    w = SMALL["tiny"]
    layer = DeviceLayer(w)
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_workspace_set_dispatch(layer.ws, 7)
    assert ei.value.status == mx.MOE_ERR_INVALID_ARG
    other = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_workspace_set_dispatch(other, mx.MOE_DISPATCH_PULL)
    assert ei.value.status == mx.MOE_ERR_WORKSPACE_MISMATCH


@pytest.fixture(scope="module")
def dsv4_layer():
    w = synth.WORKLOADS["prefill_T16384_zipf"]
    return DeviceLayer(w, max_tokens=w.T)


@pytest.mark.parametrize("name", ["layer_T512", "prefill_T4096", "prefill_T16384_zipf"])
def test_pull_full_size(dsv4_layer, name):
    """Full DeepSeek-V4-Flash shape in the benchmark's launch configuration: the pull
    path's intermediate codes equal the bucketed path's, and sampled tokens' outputs
    meet the oracle's bar."""
    w = synth.WORKLOADS[name]
    layer = dsv4_layer
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    res = _both_modes(layer, x, ids, tw)
    got_b, inter_b, _ = res[mx.MOE_DISPATCH_BUCKETED]
    got_p, inter_p, _ = res[mx.MOE_DISPATCH_PULL]
    mx.moe_workspace_set_dispatch(layer.ws, mx.MOE_DISPATCH_BUCKETED)
    assert np.array_equal(inter_p["h_codes"], inter_b["h_codes"])
    assert np.array_equal(inter_p["h_scales"], inter_b["h_scales"])
    assert normwise_rel_err(oracle.bf16_bits_to_f64(got_p), oracle.bf16_bits_to_f64(got_b)) <= 1e-3
    rng = np.random.default_rng(17)
    tokens = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 3, replace=False)]))
    sub_ids, experts = compact_problem(ids, tokens)
    Wc = oracle_expert_weights(w, experts)
    ref = oracle.moe(x[tokens], sub_ids, tw[tokens], *Wc)
    err = normwise_rel_err(oracle.bf16_bits_to_f64(got_p[tokens]), ref["out_f64"])
    assert err <= 2e-3

"""The layer on SM pairs (MOE_TILES_PAIR: 192-row token tiles, two SMs per item with
tcgen05 cta_group::2 MMAs of M=256) against the single-SM wide tiles and the oracle.

Pairing changes which SM stages which operand rows and how many token columns one
MMA covers, not any output element's K reduction: the gate/up accumulators and the
requantised intermediate must be bit-identical to the wide tiles', the outputs equal
up to the order of the fp32 combine reductions, and everything within the oracle's
bars.  Shapes cover partial tiles (16-row TMA boxes, one or two token scale blocks),
experts with several 192-row tiles, a 128-wide last k-block (I = 384), one expert,
and the full DeepSeek-V4-Flash prefill loads.
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
from tests.helpers import normwise_rel_err, oracle_expert_weights  # noqa: E402

pytestmark = pytest.mark.gpu

SHAPES = {
    # a few tokens per expert: one 32-row MMA, 16-row boxes, one scale block
    "tiny": synth.Workload("tiny", T=16, H=256, I=128, E=8, k=2),
    # ~175 rows per expert: one partial 192-row tile (two scale blocks); I = 384 gives
    # a 128-wide last k-block in the down projection and three gate/up slab pairs
    "ragged": synth.Workload("ragged", T=700, H=512, I=384, E=8, k=2),
    # skewed: expert 0 holds several full tiles plus a tail, the rarest a handful
    "zipf": synth.Workload("zipf", T=1024, H=256, I=256, E=32, k=4, routing="zipf",
                           outlier_frac=0.001),
    "top1": synth.Workload("top1", T=96, H=256, I=128, E=1, k=1),
}


def _run(layer, x, ids, tw, mode):
    w = layer.w
    mx.moe_workspace_set_tiles(layer.ws, mode)
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    gu = torch.full((w.T * w.k, 2 * w.I), float("nan"), dtype=torch.float32, device=device())
    mx.moe_debug_gate_up(layer.dims, layer.prepared, layer.ws, gu, w.T)
    mx.moe_check(layer.ws)
    got = layer.run(x, ids, tw)
    return (gu.cpu().numpy(), got, mx.moe_read_intermediate(layer.dims, layer.ws, w.T),
            mx.moe_read_dispatch(layer.dims, layer.ws, w.T))


@pytest.mark.parametrize("name", list(SHAPES))
def test_pair_tiles_match_wide_tiles_and_oracle(name):
    w = SHAPES[name]
    layer = DeviceLayer(w)
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    gw, ow, iw, dw = _run(layer, x, ids, tw, mx.MOE_TILES_WIDE)
    gp, op, ip, dp = _run(layer, x, ids, tw, mx.MOE_TILES_PAIR)
    assert np.all(np.isfinite(gp))
    assert np.array_equal(gp, gw)
    assert np.array_equal(ip["h_codes"], iw["h_codes"])
    assert np.array_equal(ip["h_scales"], iw["h_scales"])
    # rows differ (pair tiles start 256-row spans), each assignment's token row does not
    for key in ("x_codes", "x_scales", "counts", "slot_token"):
        assert np.array_equal(dp[key], dw[key]), key
    assert np.array_equal(dp["assign_slot"] >= 0, dw["assign_slot"] >= 0)
    ref = oracle.moe(x, ids, tw, *oracle_expert_weights(w, range(w.E)))
    assert normwise_rel_err(oracle.bf16_bits_to_f64(op), oracle.bf16_bits_to_f64(ow)) <= 1e-3
    err = normwise_rel_err(oracle.bf16_bits_to_f64(op), ref["out_f64"])
    print(name, "pair tiles: normwise err", err)
    assert err <= 2e-3


def test_pair_tiles_many_tiles_an_expert_and_repeat_calls():
    """Every token on the same three experts (eleven 192-row tiles each, the last one
    partial), two forwards on one dispatch, then a smaller batch on the same workspace:
    the per-tile counters and the accumulator reset between calls."""
    w = synth.Workload("hot3", T=2000, H=256, I=256, E=16, k=3)
    layer = DeviceLayer(w, max_tokens=w.T)
    x = synth.hidden_bf16(w)
    ids = np.tile(np.array([[3, 7, 11]], np.int32), (w.T, 1))
    _, tw = synth.routing(w)
    ref = oracle.moe(x, ids, tw, *oracle_expert_weights(w, range(w.E)))
    mx.moe_workspace_set_tiles(layer.ws, mx.MOE_TILES_PAIR)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=device())
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
    first = None
    for _ in range(2):
        mx.moe_forward(layer.dims, layer.prepared, layer.ws, out, w.T)
        mx.moe_check(layer.ws)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3
        if first is None:
            first = got
        else:
            assert normwise_rel_err(oracle.bf16_bits_to_f64(got),
                                    oracle.bf16_bits_to_f64(first)) <= 1e-3
    T2 = 333
    got2 = layer.run(x[:T2], ids[:T2], tw[:T2])
    ref2 = oracle.moe(x[:T2], ids[:T2], tw[:T2], *oracle_expert_weights(w, range(w.E)))
    assert normwise_rel_err(oracle.bf16_bits_to_f64(got2), ref2["out_f64"]) <= 2e-3


def test_pair_mode_falls_back_where_it_is_not_built():
    """H = 384 (an odd number of 128-row down slabs) and the other mma types run the
    single-SM wide tiles under MOE_TILES_PAIR, with the same results."""
    w = synth.Workload("oddslab", T=512, H=384, I=256, E=4, k=2)
    layer = DeviceLayer(w)
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    gw, ow, iw, _ = _run(layer, x, ids, tw, mx.MOE_TILES_WIDE)
    gp, op, ip, _ = _run(layer, x, ids, tw, mx.MOE_TILES_PAIR)
    assert np.array_equal(gp, gw)
    assert np.array_equal(ip["h_codes"], iw["h_codes"])
    assert normwise_rel_err(oracle.bf16_bits_to_f64(op), oracle.bf16_bits_to_f64(ow)) <= 1e-3


@pytest.fixture(scope="module")
def dsv4_pair_layer():
    w = synth.WORKLOADS["prefill_T16384_zipf"]
    layer = DeviceLayer(w, max_tokens=w.T)
    mx.moe_workspace_set_tiles(layer.ws, mx.MOE_TILES_PAIR)
    return layer


@pytest.mark.parametrize("name", ["prefill_T4096", "prefill_T16384_zipf"])
def test_pair_tiles_full_size(dsv4_pair_layer, name):
    """The DeepSeek-V4-Flash prefill loads on SM pairs, in the benchmark's launch
    configuration: dispatch bit-exact, sampled tokens' intermediates and outputs
    within the oracle's bars."""
    full_size_check(dsv4_pair_layer, synth.WORKLOADS[name], "mxf4", seed=31)

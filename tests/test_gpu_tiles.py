"""Narrow (32-row) and medium (64-row) against wide (128-row) token tiles, for every
mma type.

Smaller tiles change how token rows are grouped into MMA operands and how many stages
the layer keeps in flight, not what it computes: each output column's K reduction is
the same, so the gate/up accumulators and the requantised intermediate must be
bit-identical, the outputs equal up to the order of the fp32 combine reductions, and
both within the oracle's bars.
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
from tests.gpu_common import DeviceLayer, device, to_dev  # noqa: E402
from tests.helpers import normwise_rel_err, oracle_expert_weights, oracle_expert_weights_nvf4  # noqa: E402

pytestmark = pytest.mark.gpu

SHAPES = {
    "ragged": synth.Workload("ragged", T=700, H=512, I=384, E=8, k=2),
    "zipf": synth.Workload("zipf", T=1024, H=256, I=256, E=32, k=4, routing="zipf",
                           outlier_frac=0.001),
}
MMAS = {"mxf4": mx.MOE_MMA_MXF4xMXF4, "fp8xfp4": mx.MOE_MMA_FP8xFP4, "nvf4": mx.MOE_MMA_NVF4xNVF4}
ORACLE = {"mxf4": (oracle.moe, oracle_expert_weights), "fp8xfp4": (oracle.moe_w4a8, oracle_expert_weights),
          "nvf4": (oracle.moe_nvf4, oracle_expert_weights_nvf4)}


@pytest.mark.parametrize("mma", list(MMAS))
@pytest.mark.parametrize("name", list(SHAPES))
def test_narrow_tiles_match_wide_tiles(name, mma):
    w = SHAPES[name]
    layer = DeviceLayer(w, mma_type=MMAS[mma])
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    res = {}
    for mode in (mx.MOE_TILES_WIDE, mx.MOE_TILES_MEDIUM, mx.MOE_TILES_NARROW):
        mx.moe_workspace_set_tiles(layer.ws, mode)
        mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(ids), to_dev(tw), w.T, layer.ws)
        gu = torch.full((w.T * w.k, 2 * w.I), float("nan"), dtype=torch.float32, device=device())
        mx.moe_debug_gate_up(layer.dims, layer.prepared, layer.ws, gu, w.T)
        mx.moe_check(layer.ws)
        got = layer.run(x, ids, tw)
        res[mode] = (gu.cpu().numpy(), got, mx.moe_read_intermediate(layer.dims, layer.ws, w.T),
                     mx.moe_read_dispatch(layer.dims, layer.ws, w.T))
    gw, ow, iw, dw = res[mx.MOE_TILES_WIDE]
    layer_fn, weights = ORACLE[mma]
    ref = layer_fn(x, ids, tw, *weights(w, range(w.E)))
    for mode in (mx.MOE_TILES_MEDIUM, mx.MOE_TILES_NARROW):
        gn, on, inn, dn = res[mode]
        assert np.array_equal(gn, gw)
        assert np.array_equal(inn["h_codes"], iw["h_codes"])
        assert np.array_equal(inn["h_scales"], iw["h_scales"])
        assert np.array_equal(dn["x_codes"], dw["x_codes"])
        assert np.array_equal(dn["x_scales"], dw["x_scales"])
        assert np.array_equal(dn["counts"], dw["counts"])
        assert normwise_rel_err(oracle.bf16_bits_to_f64(on), oracle.bf16_bits_to_f64(ow)) <= 1e-3
        assert normwise_rel_err(oracle.bf16_bits_to_f64(on), ref["out_f64"]) <= 2e-3


def test_tile_mode_argument_checks():
    w = synth.WORKLOADS["tiny"]
    layer = DeviceLayer(w)
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_workspace_set_tiles(layer.ws, 9)
    assert ei.value.status == mx.MOE_ERR_INVALID_ARG
    other = torch.empty(1 << 20, dtype=torch.uint8, device=device())
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_workspace_set_tiles(other, mx.MOE_TILES_NARROW)
    assert ei.value.status == mx.MOE_ERR_WORKSPACE_MISMATCH
    mx.moe_workspace_set_tiles(layer.ws, mx.MOE_TILES_AUTO)

"""The API paths of test_gpu_parity.py for the other mma types and for narrow tiles:
CUDA-graph capture and replay, the host-buffer entry point, edge token counts
(narrow and wide), invalid routing ids, and all tokens on one expert."""
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

W = synth.Workload("modes", T=300, H=256, I=256, E=16, k=3)
MMAS = {"mxf4": mx.MOE_MMA_MXF4xMXF4, "fp8xfp4": mx.MOE_MMA_FP8xFP4, "nvf4": mx.MOE_MMA_NVF4xNVF4}
ORACLE = {"mxf4": (oracle.moe, oracle_expert_weights),
          "fp8xfp4": (oracle.moe_w4a8, oracle_expert_weights),
          "nvf4": (oracle.moe_nvf4, oracle_expert_weights_nvf4)}
_cache = {}


def _setup(mma):
    if mma not in _cache:
        layer_fn, weights = ORACLE[mma]
        _cache[mma] = (DeviceLayer(W, mma_type=MMAS[mma]), layer_fn, weights(W, range(W.E)))
    return _cache[mma]


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("mma", list(MMAS))
def test_graph_replay_and_host_path(mma):
    layer, layer_fn, Wts = _setup(mma)
    x = synth.hidden_bf16(W)
    ids, tw = synth.routing(W)
    ref = layer_fn(x, ids, tw, *Wts)
    eager = layer.run(x, ids, tw)
    assert normwise_rel_err(oracle.bf16_bits_to_f64(eager), ref["out_f64"]) <= 2e-3
    xd, idd, twd = to_dev(x), to_dev(ids), to_dev(tw)
    out = torch.empty((W.T, W.H), dtype=torch.bfloat16, device=device())
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        mx.moe_pre_dispatch(layer.dims, xd, idd, twd, W.T, layer.ws, s)
        mx.moe_forward(layer.dims, layer.prepared, layer.ws, out, W.T, s)
    for _ in range(2):
        out.fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        mx.moe_check(layer.ws, s)
        assert normwise_rel_err(oracle.bf16_bits_to_f64(_bits(out)), oracle.bf16_bits_to_f64(eager)) <= 1e-3
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    oh = torch.empty((W.T, W.H), dtype=torch.int16).pin_memory()
    mx.moe_run_host(layer.dims, layer.prepared, layer.ws, xh, torch.from_numpy(ids).pin_memory(),
                    torch.from_numpy(tw).pin_memory(), oh, W.T)
    assert normwise_rel_err(oracle.bf16_bits_to_f64(oh.numpy().view(np.uint16)), ref["out_f64"]) <= 2e-3


@pytest.mark.parametrize("tiles", [mx.MOE_TILES_NARROW, mx.MOE_TILES_WIDE])
@pytest.mark.parametrize("mma", list(MMAS))
def test_edge_token_counts_and_one_expert(mma, tiles):
    layer, layer_fn, Wts = _setup(mma)
    mx.moe_workspace_set_tiles(layer.ws, tiles)
    try:
        x = synth.hidden_bf16(W)
        ids, tw = synth.routing(W)
        for T in (1, 2, 33, 129):
            got = layer.run(x[:T], ids[:T], tw[:T])
            ref = layer_fn(x[:T], ids[:T], tw[:T], *Wts)
            assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3, T
        # every token on the same three experts: 300 rows each, many tiles an expert
        one = np.tile(np.array([[2, 7, 11]], np.int32), (W.T, 1))
        got = layer.run(x, one, tw)
        ref = layer_fn(x, one, tw, *Wts)
        assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3
    finally:
        mx.moe_workspace_set_tiles(layer.ws, mx.MOE_TILES_AUTO)


@pytest.mark.parametrize("mma", list(MMAS))
def test_invalid_ids_skipped_and_reported(mma):
    layer, layer_fn, Wts = _setup(mma)
    x = synth.hidden_bf16(W)
    ids, tw = synth.routing(W)
    bad = ids.copy()
    bad[4, 1] = -1
    bad[9, 0] = W.E + 3
    out = torch.empty((W.T, W.H), dtype=torch.bfloat16, device=device())
    mx.moe_pre_dispatch(layer.dims, to_dev(x), to_dev(bad), to_dev(tw), W.T, layer.ws)
    mx.moe_forward(layer.dims, layer.prepared, layer.ws, out, W.T)
    with pytest.raises(mx.MoeError) as ei:
        mx.moe_check(layer.ws)
    assert ei.value.status == mx.MOE_ERR_ROUTING
    ref = layer_fn(x, bad, tw, *Wts)
    assert ref["invalid_ids"] == 2
    assert normwise_rel_err(oracle.bf16_bits_to_f64(_bits(out)), ref["out_f64"]) <= 2e-3
    mx.moe_check(layer.ws)   # the flag was read and cleared

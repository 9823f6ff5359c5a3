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


@pytest.mark.parametrize("tiles", [mx.MOE_TILES_NARROW, mx.MOE_TILES_MEDIUM, mx.MOE_TILES_WIDE])
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


@pytest.mark.parametrize("mma", list(MMAS))
def test_largest_hidden_size(mma):
    """hidden = 65536, the largest the ABI takes: 32 quantiser rounds per token row
    (and, for E4M3 rows, the opt-in shared-memory limit of the quantiser)."""
    w = synth.Workload("wideH", T=24, H=65536, I=128, E=3, k=2)
    layer = DeviceLayer(w, mma_type=MMAS[mma])
    layer_fn, weights = ORACLE[mma]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    got = layer.run(x, ids, tw)
    ref = layer_fn(x, ids, tw, *weights(w, range(w.E)))
    d = mx.moe_read_dispatch(layer.dims, layer.ws, w.T)
    assert np.array_equal(d["x_codes"], np.repeat(ref["x_codes"], w.k, axis=0))
    assert np.array_equal(d["x_scales"], np.repeat(ref["x_sf"], w.k, axis=0))
    assert normwise_rel_err(oracle.bf16_bits_to_f64(got), ref["out_f64"]) <= 2e-3


def test_largest_token_count():
    """num_tokens = max_tokens = 65536 on a small layer: 262144 assignments, 32
    bucketing chunks; bucketing checked whole, outputs on sampled tokens."""
    w = synth.Workload("maxT", T=65536, H=256, I=128, E=64, k=4, routing="zipf")
    layer = DeviceLayer(w)
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    got = layer.run(x, ids, tw)
    d = mx.moe_read_dispatch(layer.dims, layer.ws, w.T)
    counts, offsets, st, sj, bad = oracle.bucket(ids, w.E)
    assert bad == 0 and np.array_equal(d["counts"], counts)
    slot = d["assign_slot"]
    for e in range(w.E):
        a_sorted = st[offsets[e]:offsets[e + 1]].astype(np.int64) * w.k + sj[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(slot[a_sorted]) == 1)
    from tests.helpers import compact_problem
    rng = np.random.default_rng(41)
    tokens = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 30, replace=False)]))
    sub_ids, experts = compact_problem(ids, tokens)
    ref = oracle.moe(x[tokens], sub_ids, tw[tokens], *oracle_expert_weights(w, experts))
    assert normwise_rel_err(oracle.bf16_bits_to_f64(got[tokens]), ref["out_f64"]) <= 2e-3

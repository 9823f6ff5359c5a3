"""GPU-side test plumbing: build a layer on the device from the seeded inputs, run it
through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import block_scaled_fp4_pre_gb300 as mx
from block_scaled_fp4_pre_gb300 import weights as mxw
import oracle
import synth
from tests.helpers import (compact_problem, normwise_rel_err, oracle_expert_weights,
                           oracle_expert_weights_nvf4)


def device():
    return torch.device("cuda:0")


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device())


class DeviceLayer:
    """Prepared weights + an initialised workspace for one workload shape."""

    def __init__(self, w: synth.Workload, seed: int = 0, max_tokens: int | None = None,
                 keep_canonical: bool = False, mma_type: int = mx.MOE_MMA_MXF4xMXF4):
        self.w = w
        self.seed = seed
        self.dims = mx.make_dims(w.H, w.I, w.E, w.k, max_tokens or w.T, mma_type)
        dev = device()
        can = mxw.quantize_experts(self.dims, lambda e, o: synth.expert_w1_f32(w, e, seed, out=o),
                                   lambda e, o: synth.expert_w2_f32(w, e, seed, out=o), dev)
        self.prepared = mxw.prepare(self.dims, can, dev)
        self.canonical = can if keep_canonical else None
        self.ws = torch.empty(mx.moe_workspace_size(self.dims), dtype=torch.uint8, device=dev)
        mx.moe_workspace_init(self.dims, self.ws)
        torch.cuda.synchronize()

    def run(self, x_bits: np.ndarray, ids: np.ndarray, tw: np.ndarray) -> np.ndarray:
        T = x_bits.shape[0]
        out = torch.empty((T, self.dims.hidden), dtype=torch.bfloat16, device=device())
        mx.moe_pre_dispatch(self.dims, to_dev(x_bits), to_dev(ids), to_dev(tw), T, self.ws)
        mx.moe_forward(self.dims, self.prepared, self.ws, out, T)
        mx.moe_check(self.ws)
        return out.view(torch.int16).cpu().numpy().view(np.uint16)


def flip_stats(got_codes, got_sf, ref_codes, ref_sf):
    """Fraction of intermediate elements whose E2M1 value differs, and whether every
    difference is a single grid step (or comes with a scale change)."""
    A = got_codes.shape[0]
    gd = oracle.dequantize(got_codes.reshape(A, -1), got_sf.reshape(A, -1))
    rd = oracle.dequantize(ref_codes.reshape(A, -1), ref_sf.reshape(A, -1))
    diff = gd != rd
    frac = float(diff.mean()) if diff.size else 0.0
    scale_diff = np.repeat(got_sf != ref_sf, 32, axis=1)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    gs = np.ldexp(1.0, got_sf.astype(np.int64) - 127).repeat(32, axis=1)
    idx_g = np.searchsorted(grid, np.abs(gd) / gs)
    idx_r = np.searchsorted(grid, np.abs(rd) / gs)
    one_step = (np.abs(idx_g - idx_r) <= 1) & (np.sign(gd) * np.sign(rd) >= 0)
    ok = bool(np.all(one_step[diff & ~scale_diff]))
    return frac, ok


def compare_full(layer: DeviceLayer, x_bits, ids, tw, got_bf16, oracle_weights):
    """Whole-layer comparison on every token: returns a dict of metrics."""
    w = layer.w
    T = x_bits.shape[0]
    ref = oracle.moe(x_bits, ids, tw, *oracle_weights, want_intermediates=True)
    g = oracle.bf16_bits_to_f64(got_bf16)
    inter = mx.moe_read_intermediate(layer.dims, layer.ws, T)
    valid = ((ids >= 0) & (ids < w.E)).reshape(-1)
    frac, one_step = flip_stats(inter["h_codes"][valid], inter["h_scales"][valid],
                                ref["h_codes"][valid], ref["h_sf"][valid])
    down = oracle.moe_down(ids, tw, oracle_weights[2], oracle_weights[3], inter["h_codes"],
                           inter["h_scales"], w.H)
    return {
        "err_f64": normwise_rel_err(g, ref["out_f64"]),
        "err_bf16": normwise_rel_err(g, oracle.bf16_bits_to_f64(ref["out_bf16"])),
        "err_own_h": normwise_rel_err(g, down["out_f64"]),
        "own_h_bf16_equal": float(np.mean(got_bf16 == down["out_bf16"])),
        "flip_frac": frac,
        "flips_one_step": one_step,
        "ref": ref,
    }


def flip_stats8(got_q, got_sf, ref_q, ref_sf):
    """Fraction of intermediate elements whose MXFP8 value differs from the oracle's,
    and whether each difference (where the scale agrees) is one E4M3 step."""
    gd = oracle.mxfp8_dequantize(got_q, got_sf)
    rd = oracle.mxfp8_dequantize(ref_q, ref_sf)
    diff = gd != rd
    same_scale = np.repeat(got_sf == ref_sf, 32, axis=1)
    # E4M3 magnitudes are ordered like their 7-bit codes: one step = codes 1 apart
    mg, mr = (got_q & 0x7F).astype(int), (ref_q & 0x7F).astype(int)
    sign_ok = ((got_q ^ ref_q) & 0x80 == 0) | (mg == 0) | (mr == 0)
    one = (np.abs(mg - mr) <= 1) & sign_ok
    return float(diff.mean()) if diff.size else 0.0, bool(np.all(one[diff & same_scale]))


def flip_stats_nv(got_c, got_s, ref_c, ref_s):
    """Fraction of intermediate elements whose NVFP4 value differs from the oracle's,
    and whether each difference (where the scale agrees) is one E2M1 step."""
    gd = oracle.nvfp4_dequantize(got_c, got_s)
    rd = oracle.nvfp4_dequantize(ref_c, ref_s)
    diff = gd != rd
    same = np.repeat(got_s == ref_s, 16, axis=1)

    def mags(c):
        lo, hi = c & 7, (c >> 4) & 7
        return np.stack([lo, hi], axis=-1).reshape(c.shape[0], -1).astype(int)

    one = np.abs(mags(got_c) - mags(ref_c)) <= 1
    return float(diff.mean()) if diff.size else 0.0, bool(np.all(one[diff & same]))


# Per activation format: the oracle's layer, its token quantiser, the intermediate
# comparison and the oracle-side weights.
FORMATS = {
    "mxf4": dict(layer=oracle.moe, quant=oracle.quantize_bf16, flips=flip_stats,
                 weights=oracle_expert_weights),
    "w4a8": dict(layer=oracle.moe_w4a8, quant=oracle.mxfp8_quantize_bf16, flips=flip_stats8,
                 weights=oracle_expert_weights),
    "nvf4": dict(layer=oracle.moe_nvf4, quant=oracle.nvfp4_quantize_bf16, flips=flip_stats_nv,
                 weights=oracle_expert_weights_nvf4),
}


def sampled_tokens(w: synth.Workload, ids: np.ndarray, n: int, seed: int) -> np.ndarray:
    """First and last token, n - 2 drawn at random, and (skewed routing) the last token
    routed to the most popular expert, whose tiles are the most numerous."""
    rng = np.random.default_rng(seed)
    tokens = np.concatenate([[0, w.T - 1], rng.choice(w.T, max(0, n - 2), replace=False)])
    if w.routing == "zipf":
        tokens = np.append(tokens, np.nonzero((ids == 0).any(1))[0][-1])
    return np.unique(tokens)


def full_size_check(layer: DeviceLayer, w: synth.Workload, fmt: str, tokens=None,
                    n_sample: int = 16, seed: int = 13, weight_cache: dict | None = None) -> dict:
    """A DeepSeek-V4-Flash-sized layer in the benchmark's launch configuration against
    the oracle:
      - bucketing (counts, every assignment's token) and every stored token row's
        codes and scales bit-exact against the oracle's quantiser;
      - the intermediate codes of the checked tokens' assignments: at most 0.1% of
        elements differ from the oracle's, each by one grid step;
      - those tokens' outputs within 2e-3 normwise of the oracle's (before its bf16
        rounding), and every output finite.
    tokens: the tokens to check (default: sampled_tokens).  weight_cache: oracle-side
    weights by expert, kept across calls."""
    F = FORMATS[fmt]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    got = layer.run(x, ids, tw)
    d = mx.moe_read_dispatch(layer.dims, layer.ws, w.T)
    counts, _, _, _, bad = oracle.bucket(ids, w.E)
    assert bad == 0 and np.array_equal(d["counts"], counts)
    assert np.array_equal(d["slot_token"], np.repeat(np.arange(w.T), w.k))
    xc, xs = F["quant"](x)
    assert np.array_equal(d["x_codes"], np.repeat(xc, w.k, axis=0)), "token codes"
    assert np.array_equal(d["x_scales"], np.repeat(xs, w.k, axis=0)), "token scales"
    del d
    if tokens is None:
        tokens = sampled_tokens(w, ids, n_sample, seed)
    tokens = np.asarray(tokens)
    sub_ids, experts = compact_problem(ids, tokens)
    if weight_cache is None:
        Wc = F["weights"](w, experts)
    else:
        missing = [int(e) for e in experts if int(e) not in weight_cache]
        if missing:
            new = F["weights"](w, missing)
            for i, e in enumerate(missing):
                weight_cache[e] = tuple(a[i] for a in new)
        Wc = tuple(np.stack([weight_cache[int(e)][i] for e in experts]) for i in range(4))
    ref = F["layer"](x[tokens], sub_ids, tw[tokens], *Wc, want_intermediates=True)
    inter = mx.moe_read_intermediate(layer.dims, layer.ws, w.T)
    rows = (tokens[:, None] * w.k + np.arange(w.k)[None, :]).reshape(-1)
    frac, one_step = F["flips"](inter["h_codes"][rows], inter["h_scales"][rows],
                                ref["h_codes"], ref["h_sf"])
    g = oracle.bf16_bits_to_f64(got)
    err = normwise_rel_err(g[tokens], ref["out_f64"])
    err_bf16 = normwise_rel_err(g[tokens], oracle.bf16_bits_to_f64(ref["out_bf16"]))
    print(f"{w.name} [{fmt}] tokens checked {len(tokens)}, assignments {len(rows)}, "
          f"intermediate flip rate {frac:.3e} (one-step: {one_step}), normwise err {err:.3e} "
          f"(vs bf16-rounded oracle {err_bf16:.3e})")
    assert frac <= 1e-3 and one_step
    assert err <= 2e-3
    assert np.all(np.isfinite(g))
    return {"flip_frac": frac, "err": err, "err_bf16": err_bf16, "tokens": len(tokens)}

"""GPU-side test plumbing: build a layer on the device from the seeded inputs, run it
through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import block_scaled_fp4_pre_gb300 as mx
from block_scaled_fp4_pre_gb300 import weights as mxw
import oracle
import synth
from tests.helpers import normwise_rel_err, oracle_expert_weights


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

"""Shared test helpers: oracle-side weight preparation and error metrics."""
from __future__ import annotations

import numpy as np

import oracle
import synth


def oracle_expert_weights(w: synth.Workload, experts, seed: int = 0):
    """Canonical MXFP4 weights for the listed experts, quantised by the oracle from the
    synthetic fp32 draws.  Returns (w1_codes, w1_sf, w2_codes, w2_sf) stacked in the
    order of `experts`."""
    w1c, w1s, w2c, w2s = [], [], [], []
    for e in experts:
        c, s = oracle.quantize_f32(synth.expert_w1_f32(w, int(e), seed))
        w1c.append(c)
        w1s.append(s)
        c, s = oracle.quantize_f32(synth.expert_w2_f32(w, int(e), seed))
        w2c.append(c)
        w2s.append(s)
    return np.stack(w1c), np.stack(w1s), np.stack(w2c), np.stack(w2s)


def oracle_expert_weights_nvf4(w: synth.Workload, experts, seed: int = 0):
    """As oracle_expert_weights, quantised to NVFP4 (E4M3 scale per 16 elements)."""
    w1c, w1s, w2c, w2s = [], [], [], []
    for e in experts:
        c, s = oracle.nvfp4_quantize_f32(synth.expert_w1_f32(w, int(e), seed))
        w1c.append(c)
        w1s.append(s)
        c, s = oracle.nvfp4_quantize_f32(synth.expert_w2_f32(w, int(e), seed))
        w2c.append(c)
        w2s.append(s)
    return np.stack(w1c), np.stack(w1s), np.stack(w2c), np.stack(w2s)


def normwise_rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def compact_problem(ids: np.ndarray, tokens):
    """Restrict a routing to a token subset and relabel the experts it touches 0..U-1.
    Returns (sub_ids, experts) with experts[new_label] = original expert."""
    sub = ids[np.asarray(tokens)]
    experts = np.unique(sub[(sub >= 0)])
    remap = {int(e): i for i, e in enumerate(experts)}
    new = np.vectorize(lambda e: remap.get(int(e), -1))(sub).astype(np.int32)
    return new, experts


def untile_codes(flat: np.ndarray, rows: int, K: int, kb_bytes: int = 128) -> np.ndarray:
    """Row-major [rows, K/2] codes from the library's k-block tiles: the 128 rows of a
    weight slab over one k-block of kb_bytes packed bytes are contiguous, and a short
    last k-block is zero-padded to full width (asserted here)."""
    nkb = -(-K // (2 * kb_bytes))
    t = flat.reshape(rows // 128, nkb, 128, kb_bytes).transpose(0, 2, 1, 3).reshape(rows, nkb * kb_bytes)
    assert not t[:, K // 2:].any(), "padding of the last k-block is not zero"
    return t[:, :K // 2]

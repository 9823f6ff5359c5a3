"""Pins of the fp8xfp4 (W4A8) oracle layer.

The W4A8 layer shares its weights, bucketing, SwiGLU reading and combine with the
W4A4 layer and differs in the activation format (MXFP8: E4M3 values, one UE8M0
scale per 32) and the gate/up interleave (gran=8).  Each test checks one part of it
against something that does not come from the W4A8 code itself: a hand-written
fixture, the pages' own stacking rule, the already pinned W4A4 layer on inputs that
both activation grids hold exactly, exact rational sums, and a dense MLP.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from tests.helpers import oracle_expert_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tiny_weights(H, I, E, seed):
    w = synth.Workload("pin8", T=1, H=H, I=I, E=E, k=1)
    return oracle_expert_weights(w, range(E), seed)


def test_gran8_interleave_golden_stack_rule_and_bijection():
    with open(os.path.join(GOLDEN, "interleave_gran8_I16.txt")) as f:
        want = [int(l) for l in f if l.strip() and not l.startswith("#")]
    assert list(oracle.interleave_source_rows(16, gran=8)) == want
    for I in (16, 64, 2048):
        src = oracle.interleave_source_rows(I, gran=8)
        # the pages' rule for gran=8: stack gate and up chunks of 8 along a new axis
        rows = np.arange(2 * I)
        gate = rows[:I].reshape(I // 8, 8)
        up = rows[I:].reshape(I // 8, 8)
        assert np.array_equal(src, np.stack([gate, up], axis=1).reshape(-1))
        assert sorted(src.tolist()) == list(range(2 * I))
    # and it differs from the gran=16 even/odd map
    assert not np.array_equal(oracle.interleave_source_rows(64, gran=8),
                              oracle.interleave_source_rows(64, gran=16))


def test_mxfp8_f32_path_matches_bf16_path_and_torch_cast():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((6, 256)) * np.exp(rng.uniform(-6, 6, (6, 1)))).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)          # bf16 values, exact in fp32
    xb = (bits.astype(np.uint32) << 16).view(np.float32)
    q32, s32 = oracle.mxfp8_quantize_f32(xb)
    q16, s16 = oracle.mxfp8_quantize_bf16(bits)
    assert np.array_equal(q32, q16) and np.array_equal(s32, s16)
    # dequantised values: scale * E4M3 value, the scale a power of two; each group's
    # codes are torch's round-to-nearest cast of x / scale
    deq = oracle.mxfp8_dequantize(q32, s32)
    scale = np.exp2(s32.astype(np.float64) - 127).repeat(32, axis=1)
    ref = torch.from_numpy((xb / scale).astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(ref.view(torch.uint8).numpy(), q32)
    assert np.array_equal(deq, ref.to(torch.float64).numpy() * scale)


def _on_both_grids(rng, rows, K):
    """Values that MXFP4 and MXFP8 both hold exactly: each group of 32 is E2M1 values
    (with its maximum 6 present) times a power of two."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    v = grid[rng.integers(0, 8, (rows, K))] * rng.choice([-1.0, 1.0], (rows, K))
    v[:, ::32] = 6.0
    v *= np.exp2(rng.integers(-4, 4, (rows, K // 32))).repeat(32, axis=1)
    return v.astype(np.float32)


def test_w4a8_gate_up_equals_w4a4_when_activations_fit_both_grids():
    H, I, E, T, k = 128, 64, 3, 5, 2
    W = _tiny_weights(H, I, E, seed=12)
    rng = np.random.default_rng(12)
    x = _on_both_grids(rng, T, H)
    x_bits = (x.view(np.uint32) >> 16).astype(np.uint16)       # exact: few mantissa bits
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2], [1, 0]], np.int32)
    tw = np.full((T, k), 0.5, np.float32)
    a4 = oracle.moe(x_bits, ids, tw, *W, want_intermediates=True)
    a8 = oracle.moe_w4a8(x_bits, ids, tw, *W, want_intermediates=True)
    assert np.array_equal(oracle.dequantize(a4["x_codes"], a4["x_sf"]),
                          oracle.mxfp8_dequantize(a8["x_codes"], a8["x_sf"]))
    assert np.array_equal(a8["gate_up"], a4["gate_up"])


def test_w4a8_down_equals_w4a4_down_on_shared_intermediates():
    H, I, E, T, k = 64, 128, 3, 4, 2
    W = _tiny_weights(H, I, E, seed=13)
    rng = np.random.default_rng(13)
    h = _on_both_grids(rng, T * k, I)
    hc4, hs4 = oracle.quantize_f32(h)
    hc8, hs8 = oracle.mxfp8_quantize_f32(h)
    assert np.array_equal(oracle.dequantize(hc4, hs4), h.astype(np.float64))
    assert np.array_equal(oracle.mxfp8_dequantize(hc8, hs8), h.astype(np.float64))
    ids = np.array([[0, 1], [2, 0], [1, 1], [2, 1]], np.int32)
    tw = np.array([[0.25, 0.75], [0.5, 0.5], [0.125, 0.875], [1.0, 0.0]], np.float32)
    d4 = oracle.moe_down(ids, tw, W[2], W[3], hc4, hs4, H)
    d8 = oracle.moe_w4a8_down(ids, tw, W[2], W[3], hc8, hs8, H)
    assert np.array_equal(d8["out_f64"], d4["out_f64"])
    assert np.array_equal(d8["out_bf16"], d4["out_bf16"])


def test_w4a8_gate_up_is_exact_rational_sum():
    H, I = 64, 32
    w1c, w1s, w2c, w2s = _tiny_weights(H, I, 2, seed=14)
    x_bits = synth.hidden_bf16(synth.Workload("g8", T=2, H=H, I=I, E=2, k=1), seed=14)
    ids = np.array([[1], [0]], np.int32)
    r = oracle.moe_w4a8(x_bits, ids, np.ones((2, 1), np.float32), w1c, w1s, w2c, w2s,
                        want_intermediates=True)
    xq, xs = r["x_codes"], r["x_sf"]

    def e4m3(code):     # E4M3 from its bit fields: bias 7, subnormals at exponent 0
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        mag = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        return -mag if s else mag

    def e2m1(code):
        s, E_, M = (code >> 3) & 1, (code >> 1) & 3, code & 1
        mag = Fraction(M, 2) if E_ == 0 else Fraction(2) ** (E_ - 1) * (1 + Fraction(M, 2))
        return -mag if s else mag

    for t in range(2):
        e = ids[t, 0]
        for n in (0, 7, I, 2 * I - 1):
            s = Fraction(0)
            for kk in range(H):
                xv = e4m3(int(xq[t, kk])) * Fraction(2) ** (int(xs[t, kk // 32]) - 127)
                byte = int(w1c[e, n, kk // 2])
                wv = e2m1((byte >> 4) if kk % 2 else byte & 0xF) * Fraction(2) ** (int(w1s[e, n, kk // 32]) - 127)
                s += xv * wv
            assert Fraction(r["gate_up"][t, n]) == s


def test_w4a8_single_expert_top1_is_dense_swiglu_mlp():
    H, I, T = 128, 128, 8
    w1c, w1s, w2c, w2s = _tiny_weights(H, I, 1, seed=15)
    x_bits = synth.hidden_bf16(synth.Workload("d8", T=T, H=H, I=I, E=1, k=1), seed=15)
    ids = np.zeros((T, 1), np.int32)
    tw = np.ones((T, 1), np.float32)
    got = oracle.moe_w4a8(x_bits, ids, tw, w1c, w1s, w2c, w2s)
    xd = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize_bf16(x_bits))
    GU = xd @ oracle.dequantize(w1c[0], w1s[0]).T
    Hm = (GU[:, :I] / (1 + np.exp(-GU[:, :I])) * GU[:, I:]).astype(np.float32)
    Hd = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize_f32(Hm))
    Y = Hd @ oracle.dequantize(w2c[0], w2s[0]).T
    assert np.array_equal(got["out_f64"], Y)
    # FP8 activations: closer to the unquantised MLP than the W4A4 layer
    w = synth.Workload("d8", T=T, H=H, I=I, E=1, k=1)
    W1 = synth.expert_w1_f32(w, 0, 15).astype(np.float64)
    W2 = synth.expert_w2_f32(w, 0, 15).astype(np.float64)
    xf = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    gu = xf @ W1.T
    ref = (gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]) @ W2.T
    rel8 = np.linalg.norm(got["out_f64"] - ref) / np.linalg.norm(ref)
    rel4 = np.linalg.norm(oracle.moe(x_bits, ids, tw, w1c, w1s, w2c, w2s)["out_f64"] - ref) / np.linalg.norm(ref)
    assert rel8 < rel4 and 0.02 < rel8 < 0.4


def test_w4a8_permutation_linearity_and_invalid_ids():
    w = synth.WORKLOADS["tiny"]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    W = oracle_expert_weights(w, range(w.E))
    base = oracle.moe_w4a8(x, ids, tw, *W, want_intermediates=True)
    perm = np.random.default_rng(16).permutation(w.T)
    p = oracle.moe_w4a8(x[perm], ids[perm], tw[perm], *W)
    assert np.array_equal(p["out_f64"], base["out_f64"][perm])
    b = oracle.moe_w4a8(x, ids, tw * np.float32(2.0), *W, want_intermediates=True)
    assert np.array_equal(b["out_f64"], 2.0 * base["out_f64"])
    assert np.array_equal(b["h_codes"], base["h_codes"])
    bad = ids.copy()
    bad[2, 0] = -3
    r = oracle.moe_w4a8(x, bad, tw, *W)
    assert r["invalid_ids"] == 1
    keep = tw.copy()
    keep[2, 0] = 0.0
    assert np.array_equal(r["out_f64"], oracle.moe_w4a8(x, ids, keep, *W)["out_f64"])

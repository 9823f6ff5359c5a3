"""Pins of the NVFP4 oracle layer.

NVFP4 here: packed E2M1 elements with one unsigned E4M3 scale per 16 elements, the
scale the E4M3 value nearest to amax/6, the elements fp32(x / scale) rounded to E2M1
(ties to even, saturating at 6, sign kept).  Each test checks the oracle against
something that does not come from its own code: torch's float8 cast and an exhaustive
search for the codes, the already pinned MXFP4 layer on inputs both formats hold
exactly, exact rational sums, and a dense MLP.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from tests.helpers import oracle_expert_weights_nvf4

GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])


def _brute_codes(x32, s):
    """E2M1 codes of fp32 values x32 with scale s by exhaustive search over the grid."""
    out = []
    for v in x32:
        sign = 8 if np.signbit(v) else 0
        if s == 0:
            out.append(sign)
            continue
        a = min(abs(float(np.float32(v) / np.float32(s))), 6.0)
        d = np.abs(GRID - a)
        best = [m for m in range(8) if d[m] == d.min()]
        m = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out.append(sign | m)
    return out


def test_nvfp4_quantiser_against_torch_cast_and_brute_force():
    rng = np.random.default_rng(31)
    rows = (rng.standard_normal((48, 64)) * np.exp(rng.uniform(-9, 7, (48, 1)))).astype(np.float32)
    rows[0, :16] = 0.0                                   # zero scale, signed zeros
    rows[0, 16:32] = -1e-30
    rows[1, :16] = np.float32(6.0 * 0.5625)              # amax/6 exactly on the E4M3 grid
    rows[2, :16] = np.linspace(-300, 300, 16).astype(np.float32)
    codes, sf = oracle.nvfp4_quantize_f32(rows)
    for r in range(rows.shape[0]):
        for g in range(rows.shape[1] // 16):
            v = rows[r, g * 16:(g + 1) * 16]
            target = np.float32(np.abs(v).max()) / np.float32(6.0)
            want_sf = int(torch.tensor([float(target)], dtype=torch.float32)
                          .to(torch.float8_e4m3fn).view(torch.uint8).item())
            assert sf[r, g] == want_sf, (r, g)
            s = float(torch.tensor([want_sf], dtype=torch.uint8).view(torch.float8_e4m3fn)
                      .to(torch.float64).item())
            want = _brute_codes(v, s)
            got = [(codes[r, g * 8 + i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
            assert got == want, (r, g)
    assert sf[0, 0] == 0 and sf[0, 1] == 0
    assert all(((codes[0, 8 + i] & 0x88) == 0x88) for i in range(8))   # -tiny -> -0 codes


def test_nvfp4_bf16_path_equals_f32_path():
    x = synth.hidden_bf16(synth.Workload("n", T=8, H=256, I=128, E=1, k=1), seed=32)
    xf = synth.bf16_bits_to_f32(x)
    assert all(np.array_equal(a, b) for a, b in zip(oracle.nvfp4_quantize_bf16(x),
                                                     oracle.nvfp4_quantize_f32(xf)))


def _on_both_grids(rng, rows, K):
    """Groups of 32 whose two 16-halves both reach 6 * 2^e: MXFP4 and NVFP4 then share
    the scale 2^e and hold every value exactly."""
    v = GRID[rng.integers(0, 8, (rows, K))] * rng.choice([-1.0, 1.0], (rows, K))
    v[:, ::16] = 6.0
    v *= np.exp2(rng.integers(-5, 3, (rows, K // 32))).repeat(32, axis=1)
    return v.astype(np.float32)


def test_nvf4_layer_equals_mxfp4_layer_on_shared_grid():
    H, I, E, T, k = 128, 64, 3, 5, 2
    rng = np.random.default_rng(33)
    W4, W8 = [], []
    for K, rows in ((H, 2 * I), (I, H)):
        w = np.stack([_on_both_grids(rng, rows, K) for _ in range(E)])
        c4 = [oracle.quantize_f32(m) for m in w]
        c8 = [oracle.nvfp4_quantize_f32(m) for m in w]
        for (a, b), m in zip(c4, w):
            assert np.array_equal(oracle.dequantize(a, b), m.astype(np.float64))
        for (a, b), m in zip(c8, w):
            assert np.array_equal(oracle.nvfp4_dequantize(a, b), m.astype(np.float64))
        W4 += [np.stack([a for a, _ in c4]), np.stack([b for _, b in c4])]
        W8 += [np.stack([a for a, _ in c8]), np.stack([b for _, b in c8])]
    x = _on_both_grids(rng, T, H)
    x_bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    ids = np.array([[0, 1], [2, 0], [1, 2], [0, 2], [1, 0]], np.int32)
    tw = np.full((T, k), 0.5, np.float32)
    a = oracle.moe(x_bits, ids, tw, *W4, want_intermediates=True)
    b = oracle.moe_nvf4(x_bits, ids, tw, *W8, want_intermediates=True)
    assert np.array_equal(a["gate_up"], b["gate_up"])


def test_nvf4_gate_up_is_exact_rational_sum():
    H, I = 64, 32
    w = synth.Workload("pn", T=2, H=H, I=I, E=2, k=1)
    w1c, w1s, w2c, w2s = oracle_expert_weights_nvf4(w, range(2), 34)
    x_bits = synth.hidden_bf16(w, seed=34)
    ids = np.array([[1], [0]], np.int32)
    r = oracle.moe_nvf4(x_bits, ids, np.ones((2, 1), np.float32), w1c, w1s, w2c, w2s,
                        want_intermediates=True)

    def e2m1(code):
        s, E_, M = (code >> 3) & 1, (code >> 1) & 3, code & 1
        mag = Fraction(M, 2) if E_ == 0 else Fraction(2) ** (E_ - 1) * (1 + Fraction(M, 2))
        return -mag if s else mag

    def ue4m3(b):
        e, m = (b >> 3) & 15, b & 7
        return Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)

    def val(codes, sf, row, kk):
        byte = int(codes[row, kk // 2])
        return e2m1((byte >> 4) if kk % 2 else byte & 0xF) * ue4m3(int(sf[row, kk // 16]))

    for t in range(2):
        e = ids[t, 0]
        for n in (0, 9, I, 2 * I - 1):
            s = sum(val(r["x_codes"], r["x_sf"], t, kk) * val(w1c[e], w1s[e], n, kk) for kk in range(H))
            assert Fraction(r["gate_up"][t, n]) == s


def test_nvf4_single_expert_top1_is_dense_swiglu_mlp():
    H, I, T = 128, 128, 8
    w = synth.Workload("dn", T=T, H=H, I=I, E=1, k=1)
    w1c, w1s, w2c, w2s = oracle_expert_weights_nvf4(w, range(1), 35)
    x_bits = synth.hidden_bf16(w, seed=35)
    ids = np.zeros((T, 1), np.int32)
    tw = np.ones((T, 1), np.float32)
    got = oracle.moe_nvf4(x_bits, ids, tw, w1c, w1s, w2c, w2s)
    xd = oracle.nvfp4_dequantize(*oracle.nvfp4_quantize_bf16(x_bits))
    GU = xd @ oracle.nvfp4_dequantize(w1c[0], w1s[0]).T
    Hm = (GU[:, :I] / (1 + np.exp(-GU[:, :I])) * GU[:, I:]).astype(np.float32)
    Hd = oracle.nvfp4_dequantize(*oracle.nvfp4_quantize_f32(Hm))
    Y = Hd @ oracle.nvfp4_dequantize(w2c[0], w2s[0]).T
    assert np.array_equal(got["out_f64"], Y)
    W1 = synth.expert_w1_f32(w, 0, 35).astype(np.float64)
    W2 = synth.expert_w2_f32(w, 0, 35).astype(np.float64)
    xf = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    gu = xf @ W1.T
    ref = (gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]) @ W2.T
    rel = np.linalg.norm(got["out_f64"] - ref) / np.linalg.norm(ref)
    assert 0.03 < rel < 0.5


def test_nvf4_permutation_and_linearity():
    w = synth.WORKLOADS["tiny"]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    W = oracle_expert_weights_nvf4(w, range(w.E))
    base = oracle.moe_nvf4(x, ids, tw, *W, want_intermediates=True)
    perm = np.random.default_rng(36).permutation(w.T)
    p = oracle.moe_nvf4(x[perm], ids[perm], tw[perm], *W)
    assert np.array_equal(p["out_f64"], base["out_f64"][perm])
    b = oracle.moe_nvf4(x, ids, tw * np.float32(2.0), *W, want_intermediates=True)
    assert np.array_equal(b["out_f64"], 2.0 * base["out_f64"])
    assert np.array_equal(b["h_codes"], base["h_codes"])

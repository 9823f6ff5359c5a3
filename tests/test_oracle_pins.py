"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one step of the oracle against a definition, a closed form, an
exhaustive search, exact rational arithmetic, an invariant, a special case that
reduces to a dense MLP, or a hand-derived fixture under tests/golden/.
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import synth
from tests.helpers import oracle_expert_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# E2M1 element format

def e2m1_from_bitfields(code: int) -> Fraction:
    """E2M1 from its bit fields: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
    Normal: 2^(E-1) * (1 + M/2); subnormal (E == 0): M/2."""
    s, E, M = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = Fraction(M, 2) if E == 0 else Fraction(2) ** (E - 1) * (1 + Fraction(M, 2))
    return -mag if s else mag


def test_e2m1_grid_matches_bitfield_definition():
    for code in range(16):
        v = oracle.e2m1_value(code)
        assert Fraction(v) == e2m1_from_bitfields(code), code
        if code & 8:
            assert math.copysign(1.0, v) == -1.0  # 0x8 is -0.0


def test_e2m1_round_trip_all_codes():
    for code in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_value(code)) == code


def _brute_force_code(q: Fraction, negative: bool) -> int:
    """Nearest code by exhaustive search over the 16 codes with the input's sign;
    a tie picks the even mantissa code."""
    cands = [c for c in range(16) if bool(c & 8) == negative]
    best = min(cands, key=lambda c: (abs(e2m1_from_bitfields(c) - q), c & 1))
    return best


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(1)
    qs = list(rng.uniform(-6, 6, 3000))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for m in mids:
        for d in (0.0, 1e-12, -1e-12, 2.0 ** -40):
            qs += [m + d, -(m + d)]
    qs += [0.0, -0.0, 6.0, -6.0, 1e-300, -1e-300]
    for q in qs:
        neg = math.copysign(1.0, q) < 0
        assert oracle.e2m1_encode(q) == _brute_force_code(Fraction(q), neg), q


def test_e2m1_rounding_golden():
    with open(os.path.join(GOLDEN, "e2m1_rounding.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            q, code = line.split("->")
            assert oracle.e2m1_encode(float(q)) == int(code.strip(), 16), line


# --------------------------------------------------------------------------
# Per-32 UE8M0 scale

def _exponent_by_definition(amax: float) -> int:
    """Smallest integer e in [-127, 127] with amax <= 6 * 2^e, by exact rationals."""
    a = Fraction(amax)
    for e in range(-127, 128):
        if a <= 6 * Fraction(2) ** e:
            return e
    raise AssertionError("no exponent")


def test_mx_exponent_against_definition():
    rng = np.random.default_rng(2)
    vals = [0.0, 6.0, 3.0, 3.0000001, 12.0, 1.5, 0.75, 1e-45, 2.0 ** -149, 2.0 ** -126,
            6.0 * 2.0 ** -127, 6.0 * 2.0 ** -128, float(np.float32(3.4e38))]
    for e in range(-130, 125):
        six = 6.0 * 2.0 ** e
        vals += [six, float(np.nextafter(np.float32(six), np.float32(np.inf))),
                 float(np.nextafter(np.float32(six), np.float32(0)))]
    vals += list(np.abs(rng.standard_normal(500)) * 10.0 ** rng.uniform(-30, 30, 500))
    for v in vals:
        v = float(np.float32(v))
        if v == 0.0 or not math.isfinite(v):
            continue
        assert oracle.mx_exponent(v) == _exponent_by_definition(v), v
    assert oracle.mx_exponent(0.0) == -127


def test_quantize_groups_brute_force():
    rng = np.random.default_rng(3)
    groups = [rng.standard_normal(32) * 10.0 ** rng.uniform(-5, 5) for _ in range(40)]
    g = rng.standard_normal(32); g[7] *= 50; groups.append(g)                   # outlier
    groups.append(np.zeros(32))                                                  # all zero
    g = np.zeros(32); g[3] = -0.0; g[4] = -1e-30; groups.append(g)               # signed zeros
    groups.append(np.full(32, 6.0))                                              # amax = 6 exactly
    groups.append(np.array([6.0 * (1 + 2.0 ** -23)] + [1.0] * 31))               # just above 6
    groups.append(np.array([2.0 ** -140] * 32))                                  # subnormal
    # exact ties at every midpoint after scaling by 2^0 (amax = 6)
    groups.append(np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4))
    groups.append(-np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4) * 2.0 ** -9)
    x = np.stack(groups).astype(np.float32)
    codes, sf = oracle.quantize_f32(x)
    for r in range(x.shape[0]):
        amax = float(np.max(np.abs(x[r])))
        e = _exponent_by_definition(amax) if amax > 0 else -127
        assert sf[r, 0] == e + 127
        if amax > 0 and e > -127:
            ratio = Fraction(amax) / Fraction(2) ** e
            assert 3 < ratio <= 6   # invariant of the smallest exponent
        for i in range(32):
            byte = codes[r, i // 2]
            code = (byte >> 4) if i % 2 else (byte & 0xF)   # element 2i in the low nibble
            q = Fraction(float(x[r, i])) / Fraction(2) ** e
            neg = math.copysign(1.0, float(x[r, i])) < 0
            assert code == _brute_force_code(q, neg), (r, i)


def test_quantize_bf16_equals_quantize_of_widened_f32():
    bits = synth.hidden_bf16(synth.WORKLOADS["tiny"])
    c1, s1 = oracle.quantize_bf16(bits)
    c2, s2 = oracle.quantize_f32(synth.bf16_bits_to_f32(bits))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_dequantize_reconstructs_within_half_step():
    x = synth.normals_f32(0, 99, 64 * 256).reshape(64, 256)
    c, s = oracle.quantize_f32(x)
    d = oracle.dequantize(c, s)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, axis=1)
    # largest gap of the E2M1 grid is 2 (between 4 and 6): error <= 1 * 2^e
    assert np.all(np.abs(d - x) <= scale * 1.0 + 0.0)


# --------------------------------------------------------------------------
# bf16 rounding of the combined output

def test_bf16_round_matches_torch_on_float32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    v = (rng.standard_normal(20000) * 10.0 ** rng.uniform(-40, 38, 20000)).astype(np.float32)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3.0e38, 1e-40], np.float32)
    v = np.concatenate([v, ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(a)) for a in v], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_round_exact_ties():
    assert oracle.bf16_round(1 + 2.0 ** -8) == 0x3F80           # tie -> even (1.0)
    assert oracle.bf16_round(1 + 3 * 2.0 ** -8) == 0x3F82       # tie -> even (1 + 2^-6)
    assert oracle.bf16_round(1 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81  # just above the tie
    assert oracle.bf16_round(-0.0) == 0x8000


# --------------------------------------------------------------------------
# Layout helpers

def test_interleave_golden_and_bijection():
    with open(os.path.join(GOLDEN, "interleave_gran16_I32.txt")) as f:
        want = [int(l) for l in f if l.strip() and not l.startswith("#")]
    got = oracle.interleave_source_rows(32)
    assert list(got) == want
    for I in (16, 64, 128, 2048):
        src = oracle.interleave_source_rows(I)
        assert sorted(src.tolist()) == list(range(2 * I))       # a permutation
        inv = np.empty_like(src)
        inv[src] = np.arange(2 * I)
        canon = np.arange(2 * I) * 7 + 3
        assert np.array_equal(canon[src][inv], canon)           # inverse restores canonical


def test_scale_block_layout_golden():
    with open(os.path.join(GOLDEN, "scale_block_layout.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            lhs, rhs = line.split("->")
            if lhs.startswith("shape"):
                _, rows, K = lhs.split()
                rows, K = int(rows), int(K)
                shape = [int(v) for v in rhs.split()]
                # 4-D int32 shape [ceil(rows/128), K/128, 32, 4]; bytes = 4x its element count
                assert shape == [(rows + 127) // 128, K // 128, 32, 4]
                layout = oracle.scale_block_layout(np.zeros((rows, K // 32), np.uint8))
                assert layout.size == 4 * int(np.prod(shape))
                continue
            rows, K, r, s = (int(v) for v in lhs.split())
            assert oracle.scale_block_offset(r, s, K // 32) == int(rhs), line


def test_scale_block_layout_is_injective():
    Kc = 16
    offs = {oracle.scale_block_offset(r, s, Kc) for r in range(256) for s in range(Kc)}
    assert len(offs) == 256 * Kc and max(offs) == 256 * Kc - 1


# --------------------------------------------------------------------------
# Bucketing

def test_bucket_order_and_counts():
    ids = np.array([[2, 0], [0, 2], [1, 2], [9, -1]], np.int32)
    counts, offsets, st, sj, bad = oracle.bucket(ids, 3)
    assert counts.tolist() == [2, 1, 3] and offsets.tolist() == [0, 2, 3, 6] and bad == 2
    assert list(zip(st, sj)) == [(0, 1), (1, 0), (2, 0), (0, 0), (1, 1), (2, 1)]


# --------------------------------------------------------------------------
# Whole layer

def _tiny_weights(H, I, E, seed):
    w = synth.Workload("pin", T=1, H=H, I=I, E=E, k=1)
    return w, oracle_expert_weights(w, range(E), seed)


def _literal_layer(x_bits, ids, tw, w1c, w1s, w2c, w2s):
    """A literal per-(t, j) loop with no bucketing: dequantise, numpy matmuls,
    SwiGLU in double rounded to fp32, requantise, down projection, weighted sum."""
    T, H = x_bits.shape
    k = ids.shape[1]
    E, twoI, _ = w1c.shape
    I = twoI // 2
    xc, xs = oracle.quantize_bf16(x_bits)
    xd = oracle.dequantize(xc, xs)
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            if e < 0 or e >= E:
                continue
            W1 = oracle.dequantize(w1c[e], w1s[e])
            gu = W1 @ xd[t]
            g, u = gu[:I], gu[I:]
            h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
            hc, hs = oracle.quantize_f32(h[None, :])
            hd = oracle.dequantize(hc, hs)[0]
            y = oracle.dequantize(w2c[e], w2s[e]) @ hd
            out[t] += float(tw[t, j]) * y
    return out


def test_brute_force_tiny_moe_all_id_combinations():
    H = I = 64
    E, k, T = 3, 2, 2
    _, (w1c, w1s, w2c, w2s) = _tiny_weights(H, I, E, seed=5)
    x = synth.normals_f32(5, 7, T * H).reshape(T, H)
    x_bits = (x.view(np.uint32) >> 16).astype(np.uint16)   # truncation is fine for inputs
    tw = np.array([[0.625, 0.375], [0.25, 0.75]], np.float32)
    pairs = [p for p in itertools.permutations(range(E), 2)]
    for combo in itertools.product(pairs, repeat=T):
        ids = np.array(combo, np.int32)
        got = oracle.moe(x_bits, ids, tw, w1c, w1s, w2c, w2s)["out_f64"]
        want = _literal_layer(x_bits, ids, tw, w1c, w1s, w2c, w2s)
        assert np.array_equal(got, want), combo


def test_single_expert_top1_is_dense_swiglu_mlp():
    H, I, T = 128, 128, 8
    _, (w1c, w1s, w2c, w2s) = _tiny_weights(H, I, 1, seed=6)
    x_bits = synth.hidden_bf16(synth.Workload("d", T=T, H=H, I=I, E=1, k=1), seed=6)
    ids = np.zeros((T, 1), np.int32)
    tw = np.ones((T, 1), np.float32)        # softmax over one expert
    got = oracle.moe(x_bits, ids, tw, w1c, w1s, w2c, w2s)
    # dense MLP on whole matrices (no routing at all), same quantisation points
    xd = oracle.dequantize(*oracle.quantize_bf16(x_bits))
    GU = xd @ oracle.dequantize(w1c[0], w1s[0]).T
    Hm = (GU[:, :I] / (1 + np.exp(-GU[:, :I])) * GU[:, I:]).astype(np.float32)
    Hd = oracle.dequantize(*oracle.quantize_f32(Hm))
    Y = Hd @ oracle.dequantize(w2c[0], w2s[0]).T
    assert np.array_equal(got["out_f64"], Y)
    # and it is an FP4-level approximation of the unquantised fp64 MLP
    w = synth.Workload("d", T=T, H=H, I=I, E=1, k=1)
    W1 = synth.expert_w1_f32(w, 0, 6).astype(np.float64)
    W2 = synth.expert_w2_f32(w, 0, 6).astype(np.float64)
    xf = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    gu = xf @ W1.T
    ref = (gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]) @ W2.T
    rel = np.linalg.norm(got["out_f64"] - ref) / np.linalg.norm(ref)
    assert 0.05 < rel < 0.5   # four FP4 quantisation points, ~0.12 each


def test_gate_up_is_exact_rational_sum():
    H, I = 64, 32
    _, (w1c, w1s, w2c, w2s) = _tiny_weights(H, I, 2, seed=7)
    x_bits = synth.hidden_bf16(synth.Workload("g", T=2, H=H, I=I, E=2, k=1), seed=7)
    ids = np.array([[1], [0]], np.int32)
    r = oracle.moe(x_bits, ids, np.ones((2, 1), np.float32), w1c, w1s, w2c, w2s,
                   want_intermediates=True)
    xc, xs = oracle.quantize_bf16(x_bits)

    def exact(codes, sf, row, kk):
        byte = codes[row, kk // 2]
        code = (byte >> 4) if kk % 2 else byte & 0xF
        return e2m1_from_bitfields(int(code)) * Fraction(2) ** (int(sf[row, kk // 32]) - 127)

    for t in range(2):
        e = ids[t, 0]
        for n in (0, 5, I, 2 * I - 1):
            s = sum(exact(xc, xs, t, kk) * exact(w1c[e], w1s[e], n, kk) for kk in range(H))
            assert Fraction(r["gate_up"][t, n]) == s


def test_token_permutation_and_expert_relabel_invariance():
    w = synth.WORKLOADS["tiny"]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    W = oracle_expert_weights(w, range(w.E))
    base = oracle.moe(x, ids, tw, *W)
    perm = np.random.default_rng(8).permutation(w.T)
    p = oracle.moe(x[perm], ids[perm], tw[perm], *W)
    assert np.array_equal(p["out_bf16"], base["out_bf16"][perm])
    assert np.array_equal(p["out_f64"], base["out_f64"][perm])
    relabel = np.random.default_rng(9).permutation(w.E)   # new label of old expert e
    inv = np.argsort(relabel)
    W2 = tuple(a[inv] for a in W)                          # new expert n = old expert inv[n]
    r = oracle.moe(x, relabel[ids].astype(np.int32), tw, *W2)
    assert np.array_equal(r["out_f64"], base["out_f64"])


def test_combine_is_linear_in_routing_weights():
    w = synth.WORKLOADS["tiny"]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    W = oracle_expert_weights(w, range(w.E))
    a = oracle.moe(x, ids, tw, *W)
    b = oracle.moe(x, ids, tw * np.float32(2.0), *W)
    assert np.array_equal(b["out_f64"], 2.0 * a["out_f64"])
    # the intermediate does not depend on the routing weights (weight applied at combine)
    c = oracle.moe(x, ids, tw, *W, want_intermediates=True)
    d = oracle.moe(x, ids, tw * np.float32(0.5), *W, want_intermediates=True)
    assert np.array_equal(c["h_codes"], d["h_codes"]) and np.array_equal(c["h_sf"], d["h_sf"])


def test_invalid_ids_contribute_nothing():
    w = synth.WORKLOADS["tiny"]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    W = oracle_expert_weights(w, range(w.E))
    bad = ids.copy()
    bad[3, 1] = -1
    bad[5, 0] = w.E
    r = oracle.moe(x, bad, tw, *W)
    assert r["invalid_ids"] == 2
    tw0 = tw.copy()
    tw0[3, 1] = 0.0
    tw0[5, 0] = 0.0
    ok = ids.copy()
    ok[3, 1] = ids[3, 0] if ids[3, 0] != ids[3, 1] else ids[3, 1]
    s = oracle.moe(x, ok, tw0, *W)
    assert np.array_equal(r["out_f64"], s["out_f64"])


def test_down_projection_entry_matches_full_layer():
    w = synth.WORKLOADS["tiny"]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    W = oracle_expert_weights(w, range(w.E))
    full = oracle.moe(x, ids, tw, *W, want_intermediates=True)
    down = oracle.moe_down(ids, tw, W[2], W[3], full["h_codes"], full["h_sf"], w.H)
    assert np.array_equal(down["out_f64"], full["out_f64"])
    assert np.array_equal(down["out_bf16"], full["out_bf16"])


def test_threads_do_not_change_results():
    w = synth.WORKLOADS["tiny"]
    x = synth.hidden_bf16(w)
    ids, tw = synth.routing(w)
    W = oracle_expert_weights(w, range(w.E))
    a = oracle.moe(x, ids, tw, *W, nthreads=1)
    b = oracle.moe(x, ids, tw, *W, nthreads=5)
    assert np.array_equal(a["out_f64"], b["out_f64"])


# --------------------------------------------------------------------------
# MXFP8 producer (SGLang PR #48424, "DeepGEMM producers write FlashInfer's 128x4
# scale layout"): E4M3 values with one UE8M0 scale per 32 elements.

def _e4m3_all_values():
    return np.array([oracle.e4m3_value(c) for c in range(256)])


def test_e4m3_grid_matches_torch_float8():
    """Every E4M3 code decodes to what PyTorch's float8_e4m3fn type gives it."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    got = _e4m3_all_values()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert got[0x7E] == 448.0 and np.isnan(got[0x7F]) and got[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_and_brute_force():
    """Round to nearest E4M3, ties to the even mantissa: against PyTorch's cast and a
    brute-force nearest search, on every exact tie between neighbouring codes, on
    the codes themselves, on the subnormal range and on random values."""
    vals = _e4m3_all_values()
    pos = np.sort(vals[:0x7F])                  # 0 .. 448, finite non-negative
    # fp32 values (the producer's scaled inputs are bf16 * 2^-e, exact in fp32);
    # PyTorch casts wider types through fp32, so fp32 inputs make its cast a
    # single rounding
    ties = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    rng = np.random.default_rng(21)
    q = np.concatenate([pos.astype(np.float32), ties, np.nextafter(ties, np.float32(0)),
                        np.nextafter(ties, np.float32(1e9)),
                        rng.uniform(0, 448, 4000).astype(np.float32),
                        rng.uniform(0, 2.0 ** -5, 1000).astype(np.float32),
                        (2.0 ** rng.uniform(-12, 8.8, 2000)).astype(np.float32)])
    q = np.clip(q, 0, 448).astype(np.float64)
    q = np.concatenate([q, -q])
    got = np.array([oracle.e4m3_encode(v) for v in q])
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    # brute force: nearest finite code, ties to the even code, sign kept
    cand = np.arange(0x7F)
    for v, c in zip(q[::7], got[::7]):
        d = np.abs(vals[cand] - abs(v))
        best = cand[d == d.min()]
        want = best[best % 2 == 0][0] if len(best) > 1 else best[0]
        assert c == (want | (0x80 if np.signbit(v) else 0))


def test_mxfp8_exponent_against_definition():
    rng = np.random.default_rng(22)
    amaxes = np.concatenate([[0.0, 448.0, 448.0 * (1 + 2.0 ** -20), 224.0, 1.0, 2.0 ** -140],
                             2.0 ** rng.uniform(-130, 120, 3000)])
    for a in amaxes:
        e = oracle.mxfp8_exponent(a)
        if a == 0:
            assert e == -127
            continue
        # smallest e with a <= 448 * 2^e, within the clamp
        want = next(k for k in range(-200, 200) if a <= 448.0 * 2.0 ** k)
        assert e == max(-127, min(127, want))


def test_mxfp8_quantize_rows_against_torch_cast():
    """Whole rows: each group's scale is the definition's, and its elements are
    PyTorch's E4M3 cast of x * 2^-e; nonzero groups fill the top binade."""
    rng = np.random.default_rng(23)
    x = (rng.standard_normal((37, 256)) * 10.0 ** rng.uniform(-4, 4, (37, 1))).astype(np.float32)
    x[3, 32:64] = 0.0
    x[5, ::41] *= 300.0
    bits = (torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()).view(np.uint16)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    q, sf = oracle.mxfp8_quantize_bf16(bits)
    g = xb.reshape(37, 8, 32)
    amax = np.abs(g).max(axis=2)
    e = sf.astype(np.int64) - 127
    for r in range(37):
        for j in range(8):
            assert e[r, j] == oracle.mxfp8_exponent(amax[r, j])
            if amax[r, j] > 0:
                assert 224.0 < amax[r, j] * 2.0 ** -e[r, j] <= 448.0
    scaled = g * np.ldexp(1.0, -e)[..., None]
    ref = torch.from_numpy(scaled.reshape(37, 256)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    assert np.all(sf[3, 1] == 0)


def test_mxfp8_packed_scales_are_row_major_bytes_as_int32():
    sf = np.arange(3 * 16, dtype=np.uint8).reshape(3, 16)
    packed = oracle.mxfp8_packed_scales(sf)
    assert packed.shape == (3, 4)
    assert packed[1, 2] == (24 | 25 << 8 | 26 << 16 | 27 << 24)   # row 1 = bytes 16..31
    assert np.array_equal(packed.view(np.uint8).reshape(3, 16), sf)   # little-endian host

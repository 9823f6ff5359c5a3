// CPU oracle of the W4A4 MXFP4 mixture-of-experts expert layer.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
// benchmark's CPU-baseline leg may load this library.  The product (the CUDA
// library and its Python binding) never calls it and shares no code with it.
//
// It restates, plainly and slowly, what the layer computes, in the order the
// pages describe it:
//   * "[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4 mega-MoE (W4A4)"
//     (top, and Appendix B): a packed FP4 x FP4 (W4A4) mega-MoE kernel on a
//     DeepSeek-V4-Flash layer (hidden 4096, inter 2048, 256 experts, top-6).
//   * prhub digest of SGLang PR #37279, section "实现拆解" items 3-4 and the
//     mega_moe.py source excerpt: pre_dispatch quantises bf16 hidden states
//     to packed E2M1 with group_size=32 for mma_type "mxf4xmxf4"; the expert
//     buffer uses activation "swiglu"; the gate/up rows of the first weight
//     are interleaved with gran=16 (even/odd) for MXFP4 activations.
//   * SGLang PR #48424, "DeepGEMM producers write FlashInfer's 128x4 scale
//     layout": the 4-D int32 scale shape [ceil(rows/128), K/128, 32, 4].
//
// Readings where the pages are silent (each is listed in the design notes):
//   R1 E2M1 code s*8+m decodes to (-1)^s * {0,0.5,1,1.5,2,3,4,6}[m] (OCP MX);
//      element 2i of a row sits in the low nibble of byte i.
//   R2 The per-32 scale is 2^e with e the smallest integer such that
//      amax <= 6 * 2^e (i.e. e = ceil(log2(amax/6)) evaluated exactly),
//      clamped to [-127, 127]; amax = 0 gives e = -127.  Stored as the UE8M0
//      byte e + 127.
//   R3 Each element x becomes the E2M1 value nearest to x * 2^-e; a tie goes
//      to the code with even mantissa index; the sign bit follows x (so a
//      negative value that rounds to zero is code 0x8).
//   R4 Gate rows are the first I rows of the first weight, up rows the last I.
//   R5 Within an expert, assignments (t, j) are ordered by ascending t then j.
//   R6 h = silu(g) * u = g / (1 + exp(-g)) * u from exact g, u, rounded once to
//      fp32; h is requantised with R2/R3 over 32-groups along I (no bf16 step).
//   R7 The routing weight is applied at the combine, after the down
//      projection: out[t] = bf16_rne(sum_j w[t,j] * y[(t,j)]), summed in j
//      order in double.
//   R8 Routing ids outside [0, E) contribute nothing.
//
// Every matrix product is the plain definition: a sum over K of products of
// dequantised values, in double.  Each product is a dyadic rational with at
// most 8 significant bits, so these sums are exact for the shapes used here.

#include <cassert>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <functional>
#include <thread>
#include <vector>

namespace {

// R1: the eight E2M1 magnitudes, indexed by the 3-bit exponent/mantissa field.
const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

void parallel_for(int64_t n, int nthreads, const std::function<void(int64_t, int64_t)>& fn) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads == 1 || n == 1) {
        fn(0, n);
        return;
    }
    const int64_t parts = std::min<int64_t>(n, nthreads);
    std::vector<std::thread> pool;
    pool.reserve((size_t)parts);
    for (int64_t p = 0; p < parts; ++p) {
        const int64_t b = n * p / parts, e = n * (p + 1) / parts;
        pool.emplace_back([&fn, b, e]() { fn(b, e); });
    }
    for (auto& th : pool) th.join();
}

double bf16_bits_to_double(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

}  // namespace

extern "C" {

// R1: value of one 4-bit code.
double oracle_e2m1_value(int code) {
    const double m = kE2M1Magnitude[code & 7];
    return (code & 8) ? -m : m;
}

// R2: smallest e with amax <= 6 * 2^e, clamped to [-127, 127].
int oracle_mx_exponent(double amax) {
    assert(std::isfinite(amax) && amax >= 0.0);
    if (amax == 0.0) return -127;
    int p = 0;
    (void)std::frexp(amax, &p);  // amax = f * 2^p with f in [0.5, 1)
    int e = p - 4;               // 6 * 2^(p-4) = 0.375 * 2^p < amax: too small
    assert(amax > std::ldexp(6.0, e));
    while (amax > std::ldexp(6.0, e)) ++e;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

// R3: nearest E2M1 code to q (|q| <= 6), ties to the even mantissa index,
// sign bit taken from q.
int oracle_e2m1_encode(double q) {
    const int sign = std::signbit(q) ? 8 : 0;
    const double a = std::fabs(q);
    assert(a <= 6.0);
    int best = 0;
    double best_d = a;
    for (int m = 1; m < 8; ++m) {
        const double d = std::fabs(kE2M1Magnitude[m] - a);
        if (d < best_d || (d == best_d && (m % 2) == 0)) {
            best = m;
            best_d = d;
        }
    }
    return sign | best;
}

// Quantises one group of 32 values (R2, R3); writes 16 packed bytes and one
// scale byte.
static void quantize_group(const double* v, uint8_t* codes16, uint8_t* sf) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
    const int e = oracle_mx_exponent(amax);
    int c[32];
    for (int i = 0; i < 32; ++i) c[i] = oracle_e2m1_encode(std::ldexp(v[i], -e));
    for (int i = 0; i < 16; ++i) codes16[i] = (uint8_t)(c[2 * i] | (c[2 * i + 1] << 4));
    *sf = (uint8_t)(e + 127);
}

// Row-major fp32 [rows, K] -> codes [rows, K/2], scales [rows, K/32].
void oracle_quantize_f32(const float* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf,
                         int nthreads) {
    assert(K % 32 == 0);
    parallel_for(rows, nthreads, [&](int64_t r0, int64_t r1) {
        double v[32];
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t g = 0; g < K / 32; ++g) {
                for (int i = 0; i < 32; ++i) v[i] = (double)x[r * K + g * 32 + i];
                quantize_group(v, codes + r * (K / 2) + g * 16, sf + r * (K / 32) + g);
            }
    });
}

// Row-major bf16 bits [rows, K] -> codes, scales (bf16 widens exactly).
void oracle_quantize_bf16(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf,
                          int nthreads) {
    assert(K % 32 == 0);
    parallel_for(rows, nthreads, [&](int64_t r0, int64_t r1) {
        double v[32];
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t g = 0; g < K / 32; ++g) {
                for (int i = 0; i < 32; ++i) v[i] = bf16_bits_to_double(x[r * K + g * 32 + i]);
                quantize_group(v, codes + r * (K / 2) + g * 16, sf + r * (K / 32) + g);
            }
    });
}

// codes/scales -> double values, row-major [rows, K].
void oracle_dequantize(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t K,
                       double* out) {
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            const uint8_t byte = codes[r * (K / 2) + k / 2];
            const int code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            const int e = (int)sf[r * (K / 32) + k / 32] - 127;
            out[r * K + k] = std::ldexp(oracle_e2m1_value(code), e);
        }
}

// double -> bf16 bits, round to nearest, ties to even; overflow to infinity.
uint16_t oracle_bf16_round(double v) {
    double r;
    if (v == 0.0 || !std::isfinite(v)) {
        r = v;
    } else {
        int p = std::ilogb(v);            // |v| in [2^p, 2^(p+1))
        if (p < -126) p = -126;           // below that bf16 is subnormal: fixed quantum
        const double quantum = std::ldexp(1.0, p - 7);
        r = std::nearbyint(v / quantum) * quantum;  // default mode: ties to even
        if (std::fabs(r) >= std::ldexp(1.0, 128)) r = std::copysign(INFINITY, v);
    }
    const float f = (float)r;  // exact: r has at most 8 significant bits
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

// gran=16 gate/up interleave of the first weight, for MXFP4 activations
// (digest of PR #37279, item 4): each chunk of 16 gate rows and the matching
// 16 up rows becomes [gate even (8), up even (8), gate odd (8), up odd (8)].
// Returns the canonical row (gate rows 0..I-1, up rows I..2I-1) that lands at
// prepared row r.
int64_t oracle_interleave_source_row(int64_t r, int64_t I) {
    const int64_t c = r / 32, o = r % 32;
    if (o < 8) return c * 16 + 2 * o;
    if (o < 16) return I + c * 16 + 2 * (o - 8);
    if (o < 24) return c * 16 + 2 * (o - 16) + 1;
    return I + c * 16 + 2 * (o - 24) + 1;
}

// Byte offset of scale (row r, scale column s) in the 128x4 block layout whose
// int32 view has shape [ceil(rows/128), Kc/4, 32, 4] (PR #48424): each block of
// 128 rows x 4 scale columns is 512 contiguous bytes, row r%32 picks the 16-byte
// line, (r%128)/32 the int32 within it and s%4 the byte.  Kc = K/32.
int64_t oracle_scale_block_offset(int64_t r, int64_t s, int64_t Kc) {
    return ((r / 128) * (Kc / 4) + s / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (s % 4);
}

// R5: counts per expert, canonical offsets (exclusive prefix sum of counts)
// and, for slot p = offsets[e] + rank, the (t, j) it holds.  Returns the
// number of (t, j) whose id is outside [0, E).
int64_t oracle_bucket(const int32_t* ids, int64_t T, int64_t k, int64_t E, int64_t* counts,
                      int64_t* offsets, int32_t* slot_t, int32_t* slot_j) {
    int64_t bad = 0;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t a = 0; a < T * k; ++a) {
        if (ids[a] < 0 || ids[a] >= E) {
            ++bad;
            continue;
        }
        ++counts[ids[a]];
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    std::vector<int64_t> fill(offsets, offsets + E);
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < k; ++j) {
            const int32_t e = ids[t * k + j];
            if (e < 0 || e >= E) continue;
            const int64_t p = fill[e]++;
            slot_t[p] = (int32_t)t;
            slot_j[p] = (int32_t)j;
        }
    return bad;
}

struct oracle_shape {
    int64_t T, H, I, E, k;
};

// Grouped down projection and combine from given intermediate codes:
// y[a] = dequant(h[a]) . dequant(W2[e])^T for every valid assignment a = t*k+j,
// then R7.  Used on its own to check the down projection against any given
// intermediate, and as the tail of oracle_moe.
static void dequantize_fp8_row(const uint8_t* q, const uint8_t* sf, int64_t K, double* out);

static void down_and_combine(const oracle_shape* s, const int32_t* ids, const float* tw,
                             const uint8_t* w2_codes, const uint8_t* w2_sf, const uint8_t* h_codes,
                             const uint8_t* h_sf, double* y_out, double* out_f64,
                             uint16_t* out_bf16, int nthreads, bool h_fp8 = false) {
    const int64_t T = s->T, H = s->H, I = s->I, E = s->E, k = s->k, A = T * k;
    std::vector<int64_t> counts(E), offsets(E + 1);
    std::vector<int32_t> st(A), sj(A);
    oracle_bucket(ids, T, k, E, counts.data(), offsets.data(), st.data(), sj.data());

    std::vector<double> y((size_t)A * H, 0.0);
    std::vector<double> hdq((size_t)A * I);
    parallel_for(A, nthreads, [&](int64_t a0, int64_t a1) {
        for (int64_t a = a0; a < a1; ++a)
            if (ids[a] >= 0 && ids[a] < E) {
                if (h_fp8)
                    dequantize_fp8_row(h_codes + a * I, h_sf + a * (I / 32), I, &hdq[(size_t)a * I]);
                else
                    oracle_dequantize(h_codes + a * (I / 2), h_sf + a * (I / 32), 1, I,
                                      &hdq[(size_t)a * I]);
            }
    });
    for (int64_t e = 0; e < E; ++e) {
        if (counts[e] == 0) continue;
        parallel_for(H, nthreads, [&](int64_t n0, int64_t n1) {
            std::vector<double> wrow((size_t)I);
            for (int64_t n = n0; n < n1; ++n) {
                oracle_dequantize(w2_codes + (e * H + n) * (I / 2), w2_sf + (e * H + n) * (I / 32), 1,
                                  I, wrow.data());
                for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
                    const int64_t a = (int64_t)st[p] * k + sj[p];
                    double acc = 0.0;
                    for (int64_t i = 0; i < I; ++i) acc += hdq[(size_t)a * I + i] * wrow[i];
                    y[(size_t)a * H + n] = acc;
                }
            }
        });
    }
    if (y_out) std::memcpy(y_out, y.data(), sizeof(double) * (size_t)A * H);
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        for (int64_t t = t0; t < t1; ++t)
            for (int64_t n = 0; n < H; ++n) {
                double acc = 0.0;
                for (int64_t j = 0; j < k; ++j) {
                    const int32_t e = ids[t * k + j];
                    if (e < 0 || e >= E) continue;
                    acc += (double)tw[t * k + j] * y[(size_t)(t * k + j) * H + n];
                }
                if (out_f64) out_f64[t * H + n] = acc;
                if (out_bf16) out_bf16[t * H + n] = oracle_bf16_round(acc);
            }
    });
}

// The whole layer.  Optional outputs (nullable):
//   x_codes [T, H/2], x_sf [T, H/32]          quantised hidden states
//   gate_up [A, 2I] (double)                   g (cols 0..I-1) and u (cols I..2I-1)
//   h_codes [A, I/2], h_sf [A, I/32]           requantised intermediate
//   y [A, H] (double)                          down projection per assignment
//   out_f64 [T, H], out_bf16 [T, H]            combined output
// Assignment a = t*k + j.  Weights are canonical (un-interleaved) MXFP4:
// w1 [E, 2I, H] (gate rows then up rows), w2 [E, H, I].  Returns the number
// of ids outside [0, E).
int64_t oracle_moe(const oracle_shape* s, const uint16_t* x_bf16, const int32_t* ids,
                   const float* tw, const uint8_t* w1_codes, const uint8_t* w1_sf,
                   const uint8_t* w2_codes, const uint8_t* w2_sf, double* out_f64,
                   uint16_t* out_bf16, uint8_t* x_codes_out, uint8_t* x_sf_out, double* gate_up_out,
                   uint8_t* h_codes_out, uint8_t* h_sf_out, double* y_out, int nthreads) {
    const int64_t T = s->T, H = s->H, I = s->I, E = s->E, k = s->k, A = T * k;
    assert(H % 32 == 0 && I % 32 == 0);

    // 1. quantise the hidden states (pre_dispatch, group_size=32)
    std::vector<uint8_t> xc((size_t)T * H / 2), xs((size_t)T * H / 32);
    oracle_quantize_bf16(x_bf16, T, H, xc.data(), xs.data(), nthreads);
    if (x_codes_out) std::memcpy(x_codes_out, xc.data(), xc.size());
    if (x_sf_out) std::memcpy(x_sf_out, xs.data(), xs.size());

    // 2. bucket the assignments by expert
    std::vector<int64_t> counts(E), offsets(E + 1);
    std::vector<int32_t> st(A), sj(A);
    const int64_t bad =
        oracle_bucket(ids, T, k, E, counts.data(), offsets.data(), st.data(), sj.data());

    std::vector<double> xdq((size_t)T * H);
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        for (int64_t t = t0; t < t1; ++t)
            oracle_dequantize(&xc[(size_t)t * H / 2], &xs[(size_t)t * H / 32], 1, H, &xdq[(size_t)t * H]);
    });

    // 3. grouped gate/up projection: gu[a][n] = sum_k x[t][k] * W1[e][n][k]
    std::vector<double> gu((size_t)A * 2 * I, 0.0);
    for (int64_t e = 0; e < E; ++e) {
        if (counts[e] == 0) continue;
        parallel_for(2 * I, nthreads, [&](int64_t n0, int64_t n1) {
            std::vector<double> wrow((size_t)H);
            for (int64_t n = n0; n < n1; ++n) {
                oracle_dequantize(w1_codes + (e * 2 * I + n) * (H / 2),
                                  w1_sf + (e * 2 * I + n) * (H / 32), 1, H, wrow.data());
                for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
                    const int64_t t = st[p], a = t * k + sj[p];
                    double acc = 0.0;
                    for (int64_t kk = 0; kk < H; ++kk) acc += xdq[(size_t)t * H + kk] * wrow[kk];
                    gu[(size_t)a * 2 * I + n] = acc;
                }
            }
        });
    }
    if (gate_up_out) std::memcpy(gate_up_out, gu.data(), sizeof(double) * gu.size());

    // 4-5. SwiGLU (R6) and requantisation of h along I
    std::vector<uint8_t> hc((size_t)A * I / 2, 0), hs((size_t)A * I / 32, 0);
    parallel_for(A, nthreads, [&](int64_t a0, int64_t a1) {
        std::vector<float> h((size_t)I);
        for (int64_t a = a0; a < a1; ++a) {
            if (ids[a] < 0 || ids[a] >= E) continue;
            for (int64_t i = 0; i < I; ++i) {
                const double g = gu[(size_t)a * 2 * I + i];
                const double u = gu[(size_t)a * 2 * I + I + i];
                h[i] = (float)(g / (1.0 + std::exp(-g)) * u);
            }
            oracle_quantize_f32(h.data(), 1, I, &hc[(size_t)a * I / 2], &hs[(size_t)a * I / 32], 1);
        }
    });
    if (h_codes_out) std::memcpy(h_codes_out, hc.data(), hc.size());
    if (h_sf_out) std::memcpy(h_sf_out, hs.data(), hs.size());

    // 6-7. grouped down projection and top-k weighted combine
    down_and_combine(s, ids, tw, w2_codes, w2_sf, hc.data(), hs.data(), y_out, out_f64, out_bf16,
                     nthreads);
    return bad;
}

// Down projection + combine from caller-given intermediate codes [A, I/2],
// scales [A, I/32] (a = t*k + j).  Same arithmetic as the tail of oracle_moe.
void oracle_moe_down(const oracle_shape* s, const int32_t* ids, const float* tw,
                     const uint8_t* w2_codes, const uint8_t* w2_sf, const uint8_t* h_codes,
                     const uint8_t* h_sf, double* out_f64, uint16_t* out_bf16, int nthreads) {
    down_and_combine(s, ids, tw, w2_codes, w2_sf, h_codes, h_sf, nullptr, out_f64, out_bf16,
                     nthreads);
}

// ---------------------------------------------------------------------------
// MXFP8 producer (SGLang PR #48424, section "DeepGEMM producers write
// FlashInfer's 128x4 scale layout"): a producer hands its consumer an MXFP8 pair,
// FP8 values plus one power-of-two scale per 32 elements, the scales either
// packed four to an int32 along K or in the 4-D [ceil(rows/128), K/128, 32, 4]
// int32 layout (byte order R9), with padded rows' scales zero.
// Readings where the page is silent:
//   R13 E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent
//       field 0 holds the subnormals m/8 * 2^-6; codes 0x7F and 0xFF are NaN; the
//       largest finite magnitude is 448 (exponent field 15, mantissa 6).
//   R14 The scale is 2^e with e the smallest integer such that
//       amax <= 448 * 2^e (R2 with 448 in place of 6), clamped to [-127, 127];
//       amax = 0 gives e = -127.  Stored as the UE8M0 byte e + 127.
//   R15 Each element becomes the E4M3 value nearest to x * 2^-e, a tie going to
//       the code with even mantissa field; the sign bit follows x.
//   R16 Packed scales: word j of a row holds groups 4j..4j+3 in its bytes 0..3
//       (little endian), i.e. the row-major scale bytes read as int32.

// R13: value of one E4M3 code (NaN for 0x7F / 0xFF).
double oracle_e4m3_value(int code) {
    const int e = (code >> 3) & 15, m = code & 7;
    const double sign = (code & 0x80) ? -1.0 : 1.0;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) return sign * std::ldexp((double)m / 8.0, -6);
    return sign * std::ldexp(1.0 + (double)m / 8.0, e - 7);
}

// R14: smallest e with amax <= 448 * 2^e, clamped to [-127, 127].
int oracle_mxfp8_exponent(double amax) {
    assert(std::isfinite(amax) && amax >= 0.0);
    if (amax == 0.0) return -127;
    int p = 0;
    (void)std::frexp(amax, &p);  // amax = f * 2^p, f in [0.5, 1)
    int e = p - 10;              // 448 * 2^(p-10) = 0.4375 * 2^p < amax: too small
    assert(amax > std::ldexp(448.0, e));
    while (amax > std::ldexp(448.0, e)) ++e;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

// R15: nearest E4M3 code to q (|q| <= 448, exact in double), ties to the even
// mantissa field.  The grid is uniform within each binade, spacing 2^(E-3)
// (2^-9 for the subnormals), so rounding the quotient by that spacing to the
// nearest integer, ties to even, picks the code; a result of 16 spacings is the
// first code of the next binade.
int oracle_e4m3_encode(double q) {
    const int sign = std::signbit(q) ? 0x80 : 0;
    const double a = std::fabs(q);
    assert(a <= 448.0);
    if (a < std::ldexp(1.0, -6)) {
        const double m = std::nearbyint(a / std::ldexp(1.0, -9));   // 0..8
        return sign | (int)m;                                       // 8 = smallest normal
    }
    int x = 0;
    (void)std::frexp(a, &x);      // a in [2^(x-1), 2^x)
    int E = x - 1;                // unbiased exponent, -6..8
    double r = std::nearbyint(a / std::ldexp(1.0, E - 3));   // 8..16 spacings
    if (r == 16.0) {
        ++E;
        r = 8.0;
    }
    assert(E + 7 >= 1 && E + 7 <= 15);
    const int code = ((E + 7) << 3) | ((int)r - 8);
    assert(code <= 0x7E);
    return sign | code;
}

// bf16 bits [rows, K] -> E4M3 codes [rows, K] and scale bytes [rows, K/32]
// (R14, R15), one group of 32 at a time.
void oracle_mxfp8_quantize_bf16(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                                uint8_t* sf, int nthreads) {
    assert(K % 32 == 0);
    parallel_for(rows, nthreads, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t g = 0; g < K / 32; ++g) {
                double v[32], amax = 0.0;
                for (int i = 0; i < 32; ++i) {
                    v[i] = bf16_bits_to_double(x[r * K + g * 32 + i]);
                    assert(std::isfinite(v[i]));
                    amax = std::max(amax, std::fabs(v[i]));
                }
                const int e = oracle_mxfp8_exponent(amax);
                for (int i = 0; i < 32; ++i)
                    q[r * K + g * 32 + i] = (uint8_t)oracle_e4m3_encode(std::ldexp(v[i], -e));
                sf[r * (K / 32) + g] = (uint8_t)(e + 127);
            }
    });
}

// ---------------------------------------------------------------------------
// fp8xfp4 (W4A8) layer: FP8 activations with per-32 scales against the same
// MXFP4 weights (digest of SGLang PR #37279, items 1-4: mma_type "fp8xfp4", whose
// pre_dispatch quantises the hidden states to FP8 with quant_group_size=32, and
// whose first weight interleaves gate/up with gran=8; the W4A8 column of
// "[deepseek-v4] Bump sgl-deep-gemm ...", Appendix B).
// Readings where the pages are silent:
//   R17 Both activation quantisations of this layer (the hidden states and the
//       SwiGLU output h) are MXFP8 as in R13-R15: E4M3 values, one power-of-two
//       UE8M0 scale per 32 elements along K.
//   R18 gran=8 interleave: each chunk of 8 gate rows and the matching 8 up rows
//       becomes [gate (8), up (8)], i.e. rows [gate 0..7, up 0..7, gate 8..15, ...].
//   Everything else (R4-R8) is as in the W4A4 layer.

// R18: canonical row of the first weight that lands at prepared row r.
int64_t oracle_interleave_source_row_gran8(int64_t r, int64_t I) {
    const int64_t c = r / 16, o = r % 16;
    return o < 8 ? c * 8 + o : I + c * 8 + (o - 8);
}

// One group of 32 values -> 32 E4M3 codes and one scale byte (R14, R15).
static void mxfp8_group(const double* v, uint8_t* q32, uint8_t* sf) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
        assert(std::isfinite(v[i]));
        amax = std::max(amax, std::fabs(v[i]));
    }
    const int e = oracle_mxfp8_exponent(amax);
    for (int i = 0; i < 32; ++i) q32[i] = (uint8_t)oracle_e4m3_encode(std::ldexp(v[i], -e));
    *sf = (uint8_t)(e + 127);
}

// Row-major fp32 [rows, K] -> E4M3 codes [rows, K], scale bytes [rows, K/32].
void oracle_mxfp8_quantize_f32(const float* x, int64_t rows, int64_t K, uint8_t* q, uint8_t* sf,
                               int nthreads) {
    assert(K % 32 == 0);
    parallel_for(rows, nthreads, [&](int64_t r0, int64_t r1) {
        double v[32];
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t g = 0; g < K / 32; ++g) {
                for (int i = 0; i < 32; ++i) v[i] = (double)x[r * K + g * 32 + i];
                mxfp8_group(v, q + r * K + g * 32, sf + r * (K / 32) + g);
            }
    });
}

static void dequantize_fp8_row(const uint8_t* q, const uint8_t* sf, int64_t K, double* out) {
    for (int64_t kk = 0; kk < K; ++kk)
        out[kk] = std::ldexp(oracle_e4m3_value(q[kk]), (int)sf[kk / 32] - 127);
}

// codes [rows, K] + scales [rows, K/32] -> double values [rows, K].
void oracle_mxfp8_dequantize(const uint8_t* q, const uint8_t* sf, int64_t rows, int64_t K,
                             double* out) {
    for (int64_t r = 0; r < rows; ++r) dequantize_fp8_row(q + r * K, sf + r * (K / 32), K, out + r * K);
}

// The W4A8 layer; arguments and optional outputs as oracle_moe, except that the
// quantised activations are E4M3 codes, one byte each: x_q [T, H], h_q [A, I].
int64_t oracle_moe_w4a8(const oracle_shape* s, const uint16_t* x_bf16, const int32_t* ids,
                        const float* tw, const uint8_t* w1_codes, const uint8_t* w1_sf,
                        const uint8_t* w2_codes, const uint8_t* w2_sf, double* out_f64,
                        uint16_t* out_bf16, uint8_t* x_q_out, uint8_t* x_sf_out,
                        double* gate_up_out, uint8_t* h_q_out, uint8_t* h_sf_out, double* y_out,
                        int nthreads) {
    const int64_t T = s->T, H = s->H, I = s->I, E = s->E, k = s->k, A = T * k;
    assert(H % 32 == 0 && I % 32 == 0);

    // 1. quantise the hidden states to MXFP8 (pre_dispatch, quant_group_size=32)
    std::vector<uint8_t> xq((size_t)T * H), xs((size_t)T * H / 32);
    oracle_mxfp8_quantize_bf16(x_bf16, T, H, xq.data(), xs.data(), nthreads);
    if (x_q_out) std::memcpy(x_q_out, xq.data(), xq.size());
    if (x_sf_out) std::memcpy(x_sf_out, xs.data(), xs.size());

    // 2. bucket the assignments by expert
    std::vector<int64_t> counts(E), offsets(E + 1);
    std::vector<int32_t> st(A), sj(A);
    const int64_t bad =
        oracle_bucket(ids, T, k, E, counts.data(), offsets.data(), st.data(), sj.data());

    std::vector<double> xdq((size_t)T * H);
    oracle_mxfp8_dequantize(xq.data(), xs.data(), T, H, xdq.data());

    // 3. grouped gate/up projection against the MXFP4 first weight
    std::vector<double> gu((size_t)A * 2 * I, 0.0);
    for (int64_t e = 0; e < E; ++e) {
        if (counts[e] == 0) continue;
        parallel_for(2 * I, nthreads, [&](int64_t n0, int64_t n1) {
            std::vector<double> wrow((size_t)H);
            for (int64_t n = n0; n < n1; ++n) {
                oracle_dequantize(w1_codes + (e * 2 * I + n) * (H / 2),
                                  w1_sf + (e * 2 * I + n) * (H / 32), 1, H, wrow.data());
                for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
                    const int64_t t = st[p], a = t * k + sj[p];
                    double acc = 0.0;
                    for (int64_t kk = 0; kk < H; ++kk) acc += xdq[(size_t)t * H + kk] * wrow[kk];
                    gu[(size_t)a * 2 * I + n] = acc;
                }
            }
        });
    }
    if (gate_up_out) std::memcpy(gate_up_out, gu.data(), sizeof(double) * gu.size());

    // 4-5. SwiGLU (R6) and MXFP8 requantisation of h along I (R17)
    std::vector<uint8_t> hq((size_t)A * I, 0), hs((size_t)A * I / 32, 0);
    parallel_for(A, nthreads, [&](int64_t a0, int64_t a1) {
        std::vector<float> h((size_t)I);
        for (int64_t a = a0; a < a1; ++a) {
            if (ids[a] < 0 || ids[a] >= E) continue;
            for (int64_t i = 0; i < I; ++i) {
                const double g = gu[(size_t)a * 2 * I + i];
                const double u = gu[(size_t)a * 2 * I + I + i];
                h[i] = (float)(g / (1.0 + std::exp(-g)) * u);
            }
            oracle_mxfp8_quantize_f32(h.data(), 1, I, &hq[(size_t)a * I], &hs[(size_t)a * I / 32], 1);
        }
    });
    if (h_q_out) std::memcpy(h_q_out, hq.data(), hq.size());
    if (h_sf_out) std::memcpy(h_sf_out, hs.data(), hs.size());

    // 6-7. grouped down projection (MXFP8 h against the MXFP4 second weight) and
    // the top-k weighted combine
    down_and_combine(s, ids, tw, w2_codes, w2_sf, hq.data(), hs.data(), y_out, out_f64, out_bf16,
                     nthreads, true);
    return bad;
}

// W4A8 down projection + combine from caller-given MXFP8 intermediate codes
// [A, I] and scales [A, I/32].
void oracle_moe_w4a8_down(const oracle_shape* s, const int32_t* ids, const float* tw,
                          const uint8_t* w2_codes, const uint8_t* w2_sf, const uint8_t* h_q,
                          const uint8_t* h_sf, double* out_f64, uint16_t* out_bf16, int nthreads) {
    down_and_combine(s, ids, tw, w2_codes, w2_sf, h_q, h_sf, nullptr, out_f64, out_bf16, nthreads,
                     true);
}

// ---------------------------------------------------------------------------
// NVFP4 layer (digest of SGLang PR #37279: the motivation "nvfp4 megamoe support";
// the pages give no arithmetic for it).  Readings, each the plainest one:
//   R19 NVFP4 element format: E2M1 codes as R1, packed as R1, with one scale per 16
//       elements along K; the scale is an unsigned E4M3 value (R13 without the sign),
//       stored as its byte.  No second, per-tensor scale: the pages give none, so
//       every quantised value is code value x block scale.
//   R20 Block scale: s = the E4M3 value nearest to fp32(amax / 6) (ties to even,
//       saturating at 448), amax over the 16 elements.  Element: q = fp32(x / s)
//       (correctly rounded fp32 division), then the nearest E2M1 value, ties to the
//       even code, saturating at 6; the sign bit follows x.  A scale of zero (all 16
//       values below the smallest E4M3 step) makes every code a signed zero.
//   R21 Activations (hidden states and the SwiGLU output h) and both weights use
//       R19/R20; the first weight's gate/up rows use the gran=16 interleave of FP4
//       activations.  Bucketing, SwiGLU (R6) and combine (R7) as before.

// R20 on one group of 16 fp32 values: 8 packed code bytes and one scale byte.
static void nvfp4_group(const float* v, uint8_t* codes8, uint8_t* sf) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        assert(std::isfinite(v[i]));
        amax = std::max(amax, std::fabs(v[i]));
    }
    const float target = amax / 6.0f;                       // fp32, correctly rounded
    const int sbyte = oracle_e4m3_encode(std::min((double)target, 448.0)) & 0x7F;
    const double s = oracle_e4m3_value(sbyte);
    int c[16];
    for (int i = 0; i < 16; ++i) {
        const int sign = std::signbit(v[i]) ? 8 : 0;
        if (s == 0.0) {
            c[i] = sign;
            continue;
        }
        const float q = v[i] / (float)s;                     // fp32, correctly rounded
        const double a = std::min((double)std::fabs(q), 6.0);
        c[i] = (oracle_e2m1_encode(a) & 7) | sign;
    }
    for (int i = 0; i < 8; ++i) codes8[i] = (uint8_t)(c[2 * i] | (c[2 * i + 1] << 4));
    *sf = (uint8_t)sbyte;
}

// Row-major fp32 [rows, K] -> codes [rows, K/2], scale bytes [rows, K/16].
void oracle_nvfp4_quantize_f32(const float* x, int64_t rows, int64_t K, uint8_t* codes,
                               uint8_t* sf, int nthreads) {
    assert(K % 16 == 0);
    parallel_for(rows, nthreads, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t g = 0; g < K / 16; ++g)
                nvfp4_group(x + r * K + g * 16, codes + r * (K / 2) + g * 8, sf + r * (K / 16) + g);
    });
}

// bf16 bits [rows, K] -> codes, scales (bf16 widens exactly to fp32).
void oracle_nvfp4_quantize_bf16(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes,
                                uint8_t* sf, int nthreads) {
    assert(K % 16 == 0);
    parallel_for(rows, nthreads, [&](int64_t r0, int64_t r1) {
        float v[16];
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t g = 0; g < K / 16; ++g) {
                for (int i = 0; i < 16; ++i) v[i] = (float)bf16_bits_to_double(x[r * K + g * 16 + i]);
                nvfp4_group(v, codes + r * (K / 2) + g * 8, sf + r * (K / 16) + g);
            }
    });
}

static void dequantize_nvfp4_row(const uint8_t* codes, const uint8_t* sf, int64_t K, double* out) {
    for (int64_t kk = 0; kk < K; ++kk) {
        const uint8_t byte = codes[kk / 2];
        const int code = (kk % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        out[kk] = oracle_e2m1_value(code) * oracle_e4m3_value(sf[kk / 16] & 0x7F);
    }
}

void oracle_nvfp4_dequantize(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t K,
                             double* out) {
    for (int64_t r = 0; r < rows; ++r)
        dequantize_nvfp4_row(codes + r * (K / 2), sf + r * (K / 16), K, out + r * K);
}

// The NVFP4 layer; arguments as oracle_moe, with every scale array one E4M3 byte per
// 16 elements: w1_sf [E, 2I, H/16], w2_sf [E, H, I/16], x_sf [T, H/16], h_sf [A, I/16].
int64_t oracle_moe_nvf4(const oracle_shape* s, const uint16_t* x_bf16, const int32_t* ids,
                        const float* tw, const uint8_t* w1_codes, const uint8_t* w1_sf,
                        const uint8_t* w2_codes, const uint8_t* w2_sf, double* out_f64,
                        uint16_t* out_bf16, uint8_t* x_codes_out, uint8_t* x_sf_out,
                        double* gate_up_out, uint8_t* h_codes_out, uint8_t* h_sf_out,
                        double* y_out, int nthreads) {
    const int64_t T = s->T, H = s->H, I = s->I, E = s->E, k = s->k, A = T * k;
    assert(H % 16 == 0 && I % 16 == 0);

    // 1. quantise the hidden states (R20)
    std::vector<uint8_t> xc((size_t)T * H / 2), xs((size_t)T * H / 16);
    oracle_nvfp4_quantize_bf16(x_bf16, T, H, xc.data(), xs.data(), nthreads);
    if (x_codes_out) std::memcpy(x_codes_out, xc.data(), xc.size());
    if (x_sf_out) std::memcpy(x_sf_out, xs.data(), xs.size());

    // 2. bucket
    std::vector<int64_t> counts(E), offsets(E + 1);
    std::vector<int32_t> st(A), sj(A);
    const int64_t bad =
        oracle_bucket(ids, T, k, E, counts.data(), offsets.data(), st.data(), sj.data());
    std::vector<double> xdq((size_t)T * H);
    oracle_nvfp4_dequantize(xc.data(), xs.data(), T, H, xdq.data());

    // 3. grouped gate/up projection
    std::vector<double> gu((size_t)A * 2 * I, 0.0);
    for (int64_t e = 0; e < E; ++e) {
        if (counts[e] == 0) continue;
        parallel_for(2 * I, nthreads, [&](int64_t n0, int64_t n1) {
            std::vector<double> wrow((size_t)H);
            for (int64_t n = n0; n < n1; ++n) {
                dequantize_nvfp4_row(w1_codes + (e * 2 * I + n) * (H / 2),
                                     w1_sf + (e * 2 * I + n) * (H / 16), H, wrow.data());
                for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
                    const int64_t t = st[p], a = t * k + sj[p];
                    double acc = 0.0;
                    for (int64_t kk = 0; kk < H; ++kk) acc += xdq[(size_t)t * H + kk] * wrow[kk];
                    gu[(size_t)a * 2 * I + n] = acc;
                }
            }
        });
    }
    if (gate_up_out) std::memcpy(gate_up_out, gu.data(), sizeof(double) * gu.size());

    // 4-5. SwiGLU (R6) and NVFP4 requantisation of h (R20)
    std::vector<uint8_t> hc((size_t)A * I / 2, 0), hs((size_t)A * I / 16, 0);
    parallel_for(A, nthreads, [&](int64_t a0, int64_t a1) {
        std::vector<float> h((size_t)I);
        for (int64_t a = a0; a < a1; ++a) {
            if (ids[a] < 0 || ids[a] >= E) continue;
            for (int64_t i = 0; i < I; ++i) {
                const double g = gu[(size_t)a * 2 * I + i];
                const double u = gu[(size_t)a * 2 * I + I + i];
                h[i] = (float)(g / (1.0 + std::exp(-g)) * u);
            }
            oracle_nvfp4_quantize_f32(h.data(), 1, I, &hc[(size_t)a * I / 2], &hs[(size_t)a * I / 16], 1);
        }
    });
    if (h_codes_out) std::memcpy(h_codes_out, hc.data(), hc.size());
    if (h_sf_out) std::memcpy(h_sf_out, hs.data(), hs.size());

    // 6-7. grouped down projection and combine
    std::vector<double> y((size_t)A * H, 0.0);
    std::vector<double> hdq((size_t)A * I);
    for (int64_t a = 0; a < A; ++a)
        if (ids[a] >= 0 && ids[a] < E)
            dequantize_nvfp4_row(&hc[(size_t)a * I / 2], &hs[(size_t)a * I / 16], I, &hdq[(size_t)a * I]);
    for (int64_t e = 0; e < E; ++e) {
        if (counts[e] == 0) continue;
        parallel_for(H, nthreads, [&](int64_t n0, int64_t n1) {
            std::vector<double> wrow((size_t)I);
            for (int64_t n = n0; n < n1; ++n) {
                dequantize_nvfp4_row(w2_codes + (e * H + n) * (I / 2), w2_sf + (e * H + n) * (I / 16),
                                     I, wrow.data());
                for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
                    const int64_t a = (int64_t)st[p] * k + sj[p];
                    double acc = 0.0;
                    for (int64_t i = 0; i < I; ++i) acc += hdq[(size_t)a * I + i] * wrow[i];
                    y[(size_t)a * H + n] = acc;
                }
            }
        });
    }
    if (y_out) std::memcpy(y_out, y.data(), sizeof(double) * y.size());
    parallel_for(T, nthreads, [&](int64_t t0, int64_t t1) {
        for (int64_t t = t0; t < t1; ++t)
            for (int64_t n = 0; n < H; ++n) {
                double acc = 0.0;
                for (int64_t j = 0; j < k; ++j) {
                    const int32_t e = ids[t * k + j];
                    if (e < 0 || e >= E) continue;
                    acc += (double)tw[t * k + j] * y[(size_t)(t * k + j) * H + n];
                }
                if (out_f64) out_f64[t * H + n] = acc;
                if (out_bf16) out_bf16[t * H + n] = oracle_bf16_round(acc);
            }
    });
    return bad;
}

}  // extern "C"

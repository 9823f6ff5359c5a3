/*
 * Seeded synthetic inputs for the W4A4 MXFP4 mixture-of-experts layer.
 *
 * This file draws the random tensors that both the CPU oracle and the CUDA
 * path consume: bf16 hidden states, top-k routing (uniform or Zipf), routing
 * weights and fp32 expert weights.  It contains none of the layer's own
 * arithmetic: no quantisation, no matrix product, no activation.
 *
 * Every value is a pure function of (seed, stream, index), so any slice of
 * any tensor can be regenerated on its own (for example the weights of the
 * few experts a sampled token touches) and multi-threaded generation gives
 * the same bytes as single-threaded generation.
 *
 * Generator: splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) evaluated at counter positions, uniforms
 * from its top 53 bits, normals by the Box-Muller transform (Box and
 * Muller, 1958) in double precision.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t splitmix64_at(uint64_t state) {
    uint64_t z = state + GOLDEN_GAMMA;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of one named stream of one seed. */
static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return splitmix64_at(splitmix64_at(seed) ^ (stream * 0xD1B54A32D192ED03ULL));
}

/* The i-th 64-bit draw of a stream. */
static inline uint64_t draw_u64(uint64_t key, uint64_t i) {
    return splitmix64_at(key + i * GOLDEN_GAMMA);
}

/* Uniform in (0, 1]: top 53 bits, shifted away from zero. */
static inline double draw_unit_open0(uint64_t key, uint64_t i) {
    return (double)((draw_u64(key, i) >> 11) + 1) * 0x1.0p-53;
}

/* Uniform in [0, 1). */
static inline double draw_unit(uint64_t key, uint64_t i) {
    return (double)(draw_u64(key, i) >> 11) * 0x1.0p-53;
}

/* Standard normal number `i` of a stream (Box-Muller pair i/2). */
static inline double draw_normal(uint64_t key, uint64_t i) {
    const uint64_t pair = i >> 1;
    const double u1 = draw_unit_open0(key, 2 * pair);
    const double u2 = draw_unit(key, 2 * pair + 1);
    const double r = sqrt(-2.0 * log(u1));
    const double ang = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(ang) : r * cos(ang);
}

/* Integer in [0, n) from one draw (multiply-shift on the top 32 bits). */
static inline uint32_t draw_below(uint64_t key, uint64_t i, uint32_t n) {
    const uint64_t r = draw_u64(key, i) >> 32;
    return (uint32_t)((r * (uint64_t)n) >> 32);
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs). */
static inline uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------------- */
/* Threaded fill helpers                                                   */

typedef struct {
    uint64_t key, first, count;
    double scale;
    void *out;
    int kind; /* 0: f32, 1: bf16 */
} fill_job;

static inline void store_value(const fill_job *j, uint64_t t, double v) {
    if (j->kind == 0)
        ((float *)j->out)[t] = (float)(v * j->scale);
    else
        ((uint16_t *)j->out)[t] = f32_to_bf16_bits((float)(v * j->scale));
}

/* Fills positions first..first+count-1; both members of a Box-Muller pair
 * come from one evaluation of the transform. */
static void *fill_worker(void *arg) {
    const fill_job *j = (const fill_job *)arg;
    uint64_t t = 0;
    const uint64_t end = j->count;
    if (end > 0 && (j->first & 1)) {
        store_value(j, 0, draw_normal(j->key, j->first));
        t = 1;
    }
    for (; t + 1 < end; t += 2) {
        const uint64_t pair = (j->first + t) >> 1;
        const double u1 = draw_unit_open0(j->key, 2 * pair);
        const double u2 = draw_unit(j->key, 2 * pair + 1);
        const double r = sqrt(-2.0 * log(u1));
        const double ang = 6.283185307179586476925286766559 * u2;
        store_value(j, t, r * cos(ang));
        store_value(j, t + 1, r * sin(ang));
    }
    if (t < end) store_value(j, t, draw_normal(j->key, j->first + t));
    return NULL;
}

static void fill_threaded(uint64_t key, uint64_t first, uint64_t count, double scale,
                          void *out, int kind, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (count < 65536) nthreads = 1;
    pthread_t th[256];
    fill_job jobs[256];
    const size_t esz = kind == 0 ? 4 : 2;
    uint64_t per = (count + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    per = (per + 1) & ~1ULL; /* keep Box-Muller pairs inside one worker */
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        const uint64_t b = (uint64_t)t * per;
        if (b >= count) break;
        const uint64_t c = (b + per > count) ? count - b : per;
        jobs[t].key = key;
        jobs[t].first = first + b;
        jobs[t].count = c;
        jobs[t].scale = scale;
        jobs[t].out = (char *)out + b * esz;
        jobs[t].kind = kind;
        ++used;
    }
    if (used == 1) {
        fill_worker(&jobs[0]);
        return;
    }
    for (int t = 0; t < used; ++t) pthread_create(&th[t], NULL, fill_worker, &jobs[t]);
    for (int t = 0; t < used; ++t) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------------- */
/* Public entry points                                                     */

/* out[i] = fp32(N(0,1) * sigma) for positions first..first+count-1 of a stream. */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, uint64_t count,
                      double sigma, float *out, int nthreads) {
    fill_threaded(stream_key(seed, stream), first, count, sigma, out, 0, nthreads);
}

/* out[i] = bf16_rne(fp32(N(0,1) * scale)) for positions first..first+count-1. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, uint64_t count,
                       double scale, uint16_t *out, int nthreads) {
    fill_threaded(stream_key(seed, stream), first, count, scale, out, 1, nthreads);
}

/*
 * Hidden states x [T, H] as bf16 bits: N(0,1) rounded to fp32 then bf16.
 * With n_outliers > 0, that many distinct positions, drawn uniformly without
 * replacement from the T*H positions, hold N(0,1)*outlier_mult instead.
 */
int synth_hidden_bf16(uint64_t seed, int64_t T, int64_t H, int64_t n_outliers,
                      double outlier_mult, uint16_t *out, int nthreads) {
    const uint64_t n = (uint64_t)T * (uint64_t)H;
    const uint64_t kx = stream_key(seed, 1);
    fill_threaded(kx, 0, n, 1.0, out, 1, nthreads);
    if (n_outliers <= 0) return 0;
    if ((uint64_t)n_outliers > n) return -1;
    uint8_t *taken = (uint8_t *)calloc((n + 7) / 8, 1);
    if (!taken) return -2;
    const uint64_t ko = stream_key(seed, 4);
    uint64_t draw = 0;
    int64_t placed = 0;
    while (placed < n_outliers) {
        const uint64_t hi = draw_u64(ko, draw++);
        const uint64_t pos = (uint64_t)(((unsigned __int128)hi * n) >> 64);
        if (taken[pos >> 3] & (1u << (pos & 7))) continue;
        taken[pos >> 3] |= (uint8_t)(1u << (pos & 7));
        out[pos] = f32_to_bf16_bits((float)(draw_normal(kx, pos) * outlier_mult));
        ++placed;
    }
    free(taken);
    return 0;
}

/*
 * Routing with k distinct experts per token, each k-subset equally likely
 * (partial Fisher-Yates over 0..E-1 per token), and routing weights equal to
 * the softmax of k independent N(0,1) draws, computed in double, stored fp32.
 */
int synth_routing_uniform(uint64_t seed, int64_t T, int32_t k, int32_t E, int32_t *ids,
                          float *weights) {
    if (k < 1 || k > E || E > 65536) return -1;
    const uint64_t kid = stream_key(seed, 2);
    const uint64_t kw = stream_key(seed, 3);
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!perm) return -2;
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t e = 0; e < E; ++e) perm[e] = e;
        for (int32_t j = 0; j < k; ++j) {
            const uint32_t r = draw_below(kid, (uint64_t)t * 64u + (uint64_t)j, (uint32_t)(E - j));
            const int32_t pick = j + (int32_t)r;
            const int32_t tmp = perm[j];
            perm[j] = perm[pick];
            perm[pick] = tmp;
            ids[t * k + j] = perm[j];
        }
        double z[64], mx = -INFINITY, s = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            z[j] = draw_normal(kw, (uint64_t)t * (uint64_t)k + (uint64_t)j);
            if (z[j] > mx) mx = z[j];
        }
        for (int32_t j = 0; j < k; ++j) s += exp(z[j] - mx);
        for (int32_t j = 0; j < k; ++j) weights[t * k + j] = (float)(exp(z[j] - mx) / s);
    }
    free(perm);
    return 0;
}

/*
 * Skewed routing: expert e has popularity (e+1)^(-s) (Zipf, rank e+1).
 * Each token draws k distinct experts one after another without replacement,
 * each draw proportional to the popularity of the experts not yet chosen.
 * Routing weights as in synth_routing_uniform.
 */
int synth_routing_zipf(uint64_t seed, int64_t T, int32_t k, int32_t E, double s, int32_t *ids,
                       float *weights) {
    if (k < 1 || k > E || k > 64) return -1;
    const uint64_t kz = stream_key(seed, 5);
    const uint64_t kw = stream_key(seed, 3);
    double *pop = (double *)malloc(sizeof(double) * (size_t)E);
    uint8_t *chosen = (uint8_t *)malloc((size_t)E);
    if (!pop || !chosen) {
        free(pop);
        free(chosen);
        return -2;
    }
    double total = 0.0;
    for (int32_t e = 0; e < E; ++e) {
        pop[e] = pow((double)(e + 1), -s);
        total += pop[e];
    }
    for (int64_t t = 0; t < T; ++t) {
        memset(chosen, 0, (size_t)E);
        double remaining = total;
        for (int32_t j = 0; j < k; ++j) {
            double u = draw_unit(kz, (uint64_t)t * 64u + (uint64_t)j) * remaining;
            int32_t pick = -1, last = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (chosen[e]) continue;
                last = e;
                if (u < pop[e]) {
                    pick = e;
                    break;
                }
                u -= pop[e];
            }
            if (pick < 0) pick = last; /* rounding at the very end of the scan */
            chosen[pick] = 1;
            remaining -= pop[pick];
            ids[t * k + j] = pick;
        }
        double z[64], mx = -INFINITY, sum = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            z[j] = draw_normal(kw, (uint64_t)t * (uint64_t)k + (uint64_t)j);
            if (z[j] > mx) mx = z[j];
        }
        for (int32_t j = 0; j < k; ++j) sum += exp(z[j] - mx);
        for (int32_t j = 0; j < k; ++j) weights[t * k + j] = (float)(exp(z[j] - mx) / sum);
    }
    free(pop);
    free(chosen);
    return 0;
}

/*
 * fp32 weights of one expert: rows x cols values N(0, sigma) in row-major
 * order, where `which` is 1 for the gate/up projection [2I, H] and 2 for the
 * down projection [H, I].  first_row/num_rows select a slice of rows.
 */
void synth_expert_weights_f32(uint64_t seed, int32_t which, int32_t expert, int64_t cols,
                              int64_t first_row, int64_t num_rows, double sigma, float *out,
                              int nthreads) {
    const uint64_t stream = (which == 1 ? 0x100000ULL : 0x200000ULL) + (uint64_t)expert;
    fill_threaded(stream_key(seed, stream), (uint64_t)first_row * (uint64_t)cols,
                  (uint64_t)num_rows * (uint64_t)cols, sigma, out, 0, nthreads);
}

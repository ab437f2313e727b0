/*
 * Seeded synthetic inputs for the sparse MoE layer.
 *
 * This module draws numbers and nothing else: it holds none of the layer's
 * arithmetic (no routing, no quantisation, no GEMM).  Both the CUDA path and
 * the oracle take their inputs from here.
 *
 * Generator (fixed by this file, reproduced bit for bit on every IEEE-754
 * platform; build with -ffp-contract=off so no multiply-add is fused):
 *   - SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014) in counter form: the i-th 64-bit draw of a
 *     stream with key K is mix(K + (i+1)*0x9E3779B97F4A7C15).
 *   - One stream per (seed, tensor tag, major index, attempt); the major
 *     index is the row of x / router_w or the expert of a weight tensor.
 *   - Uniform u = ((z >> 11) + 1) * 2^-53, in (0, 1].
 *   - Normal pairs by Box-Muller (Box & Muller 1958): element 2p and 2p+1
 *     of a stream are r*cos(t) and r*sin(t), r = sqrt(-2 ln u1),
 *     t = 2*pi*u2, with u1, u2 the draws 2p and 2p+1.
 *   - ln is computed here from frexp and the atanh series
 *     ln m = 2*atanh((m-1)/(m+1)); cos/sin from their Taylor series after
 *     an exact quarter-turn reduction.  Only +, -, *, / and sqrt are used,
 *     all correctly rounded, so x86-64 and aarch64 produce identical bits.
 *   - A value is sigma * z in double, rounded to fp32 (round to nearest
 *     even); bf16 tensors round that fp32 once more to nearest even.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_stream_key(uint64_t seed, uint32_t tag, uint64_t major, uint32_t attempt) {
    uint64_t k = sm_mix(seed + GOLDEN);
    k = sm_mix(k + ((uint64_t)tag + 1) * GOLDEN);
    k = sm_mix(k + (major + 1) * GOLDEN);
    k = sm_mix(k + ((uint64_t)attempt + 1) * GOLDEN);
    return k;
}

uint64_t synth_draw_u64(uint64_t key, uint64_t i) { return sm_mix(key + (i + 1) * GOLDEN); }

static double uniform01(uint64_t z) { return (double)((z >> 11) + 1) * (1.0 / 9007199254740992.0); }

/* natural log of a positive finite double */
double synth_ln(double x) {
    const double SQRT2 = 1.4142135623730951;
    const double LN2 = 0.6931471805599453;
    int e;
    double m = frexp(x, &e); /* x = m * 2^e, m in [0.5, 1) -- exact */
    m *= 2.0;
    e -= 1;                  /* m in [1, 2) */
    if (m > SQRT2) {
        m *= 0.5;
        e += 1;
    }
    double s = (m - 1.0) / (m + 1.0);
    double s2 = s * s;
    double term = s, sum = s;
    for (int n = 1; n <= 13; ++n) {
        term = term * s2;
        sum = sum + term / (double)(2 * n + 1);
    }
    return 2.0 * sum + (double)e * LN2;
}

/* cos and sin of 2*pi*u for u in (0, 1] */
static void cos_sin_turn(double u, double* c_out, double* s_out) {
    const double HALF_PI = 1.5707963267948966;
    double t = 4.0 * u; /* exact */
    int q = (int)t;
    double f = t - (double)q; /* exact, [0, 1) */
    double a = f * HALF_PI;
    double a2 = a * a;
    double sn = a, ts = a, cs = 1.0, tc = 1.0;
    for (int n = 1; n <= 13; ++n) {
        ts = ts * (-a2 / (double)((2 * n) * (2 * n + 1)));
        sn = sn + ts;
        tc = tc * (-a2 / (double)((2 * n - 1) * (2 * n)));
        cs = cs + tc;
    }
    switch (q & 3) {
        case 0: *c_out = cs; *s_out = sn; break;
        case 1: *c_out = -sn; *s_out = cs; break;
        case 2: *c_out = -cs; *s_out = -sn; break;
        default: *c_out = sn; *s_out = -cs; break;
    }
}

/* standard normal element i of stream key */
double synth_normal_at(uint64_t key, uint64_t i) {
    uint64_t p = i >> 1;
    double u1 = uniform01(synth_draw_u64(key, 2 * p));
    double u2 = uniform01(synth_draw_u64(key, 2 * p + 1));
    double r = sqrt(-2.0 * synth_ln(u1));
    double c, s;
    cos_sin_turn(u2, &c, &s);
    return (i & 1) ? r * s : r * c;
}

uint16_t synth_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* n elements [start, start+n) of one stream, as fp32 (out_f32) or bf16 (out_bf16) */
void synth_fill(uint64_t seed, uint32_t tag, uint64_t major, uint32_t attempt, uint64_t start, uint64_t n,
                double sigma, float* out_f32, uint16_t* out_bf16) {
    uint64_t key = synth_stream_key(seed, tag, major, attempt);
    uint64_t i = start, end = start + n;
    while (i < end) {
        uint64_t p = i >> 1;
        double u1 = uniform01(synth_draw_u64(key, 2 * p));
        double u2 = uniform01(synth_draw_u64(key, 2 * p + 1));
        double r = sqrt(-2.0 * synth_ln(u1));
        double c, s;
        cos_sin_turn(u2, &c, &s);
        double z[2] = {r * c, r * s};
        for (int h = (int)(i & 1); h < 2 && i < end; ++h, ++i) {
            float v = (float)(sigma * z[h]);
            if (out_f32) out_f32[i - start] = v;
            if (out_bf16) out_bf16[i - start] = synth_f32_to_bf16(v);
        }
    }
}

/* ---- threaded fill of [majors, per_major] tensors (one stream per major) ---- */
typedef struct {
    uint64_t seed;
    uint32_t tag;
    const uint32_t* attempts;
    uint64_t per_major;
    double sigma;
    float* out_f32;
    uint16_t* out_bf16;
    uint64_t major_base;
    uint64_t lo, hi; /* flat element range handled by this worker */
} fill_job;

static void* fill_worker(void* arg) {
    fill_job* j = (fill_job*)arg;
    uint64_t i = j->lo;
    while (i < j->hi) {
        uint64_t m = i / j->per_major;
        uint64_t off = i - m * j->per_major;
        uint64_t n = j->per_major - off;
        if (n > j->hi - i) n = j->hi - i;
        uint32_t att = j->attempts ? j->attempts[m] : 0u;
        synth_fill(j->seed, j->tag, j->major_base + m, att, off, n, j->sigma, j->out_f32 ? j->out_f32 + i : NULL,
                   j->out_bf16 ? j->out_bf16 + i : NULL);
        i += n;
    }
    return NULL;
}

/* out[m, 0:per_major] for m in [0, majors): stream major index = major_base + m,
 * attempt = attempts[m] (or 0 when attempts is NULL). */
void synth_tensor(uint64_t seed, uint32_t tag, uint64_t major_base, uint64_t majors, uint64_t per_major,
                  const uint32_t* attempts, double sigma, float* out_f32, uint16_t* out_bf16, int nthreads) {
    uint64_t total = majors * per_major;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (total < 65536) nthreads = 1;
    pthread_t th[256];
    fill_job jobs[256];
    uint64_t chunk = (total + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    chunk = (chunk + 1) & ~(uint64_t)1;
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        uint64_t lo = (uint64_t)t * chunk, hi = lo + chunk;
        if (lo >= total) break;
        if (hi > total) hi = total;
        fill_job j = {seed, tag, attempts, per_major, sigma, out_f32, out_bf16, major_base, lo, hi};
        jobs[t] = j;
        if (nthreads == 1) {
            fill_worker(&jobs[t]);
        } else {
            pthread_create(&th[t], NULL, fill_worker, &jobs[t]);
            ++launched;
        }
    }
    for (int t = 0; t < launched; ++t) pthread_join(th[t], NULL);
}

/* Zipf-like router bias: out[e] = bf16(fp32(alpha * ln(1/(e+1)))) */
void synth_zipf_bias_bf16(int E, double alpha, uint16_t* out) {
    for (int e = 0; e < E; ++e) {
        float v = (float)(-alpha * synth_ln((double)(e + 1)));
        out[e] = synth_f32_to_bf16(v);
    }
}

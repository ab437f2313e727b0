/*
 * ORACLE for the sparse MoE layer forward -- test infrastructure only.
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * may load this file's library.  The CUDA library never calls it and shares
 * no code, header, table or constant with it.
 *
 * Plain, slow, single-threaded C: FP8 is decoded through this file's own
 * e4m3 table and every contraction is accumulated in FP64.  Each function
 * names the passage it follows.  The pages are the "GPT-OSS on Day 0" post
 * (perplexity.ai hub blog; sections on the MoE layer and on routing) and the
 * "Hosting Qwen on Blackwell" post (section "Quantization").
 *
 * Layer, as those posts state it (MLP bullets of the gpt-oss architecture
 * list, and the MoE routing / DeepGEMM bias / combine paragraphs):
 *   router logits -> top-k -> softmax over the k selected logits (expert
 *   weights kept in bf16) -> per expert: gate/up GEMM with bias on FP8 e4m3
 *   weights with 128x128 block scales, SwiGLU, down GEMM with bias ->
 *   weighted sum of the k expert outputs.
 * Readings where the posts are silent (each also listed in the design notes):
 *   - slot order: the k selected experts of a token are stored in ascending
 *     expert index; ties between equal logits go to the lower index;
 *   - activations are quantised per token per 128-wide group, s = amax/448,
 *     code = e4m3_rne_satfinite(v / s) in IEEE fp32; amax == 0 gives s = 1
 *     and all codes +0;
 *   - gate rows [0,I) and up rows [I,2I) of w13 are each zero-padded to Ip,
 *     K is zero-padded to a multiple of 128, scales are taken over the
 *     padded 128x128 block;
 *   - routing weights: softmax in fp64, rounded to fp32, then to bf16;
 *   - h = silu(gate)*up in fp64, rounded to fp32, then requantised like x;
 *   - b13 is added before SwiGLU, b2 before the routing-weight scale;
 *   - output: the fp64 sum over the k slots, rounded once to bf16.
 * Parity pins: see tests/test_oracle_pins.py (format table, brute force,
 * invariants, hand-worked example).  Parity unpinned: whether these readings
 * are what the posts' production system did.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 / fp32 helpers                                                */
/* ------------------------------------------------------------------ */

static double bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* fp32 -> bf16, round to nearest even */
uint16_t oracle_bf16_from_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* fp64 -> bf16 in one rounding step (nearest, ties to even).
 * bf16 has 8 significant bits and the fp32 exponent range. */
uint16_t oracle_bf16_from_f64(double d) {
    if (isnan(d)) return 0x7fc0;
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    double a = fabs(d);
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex); /* a in [2^(ex-1), 2^ex) */
    int ue = ex - 8;
    if (ue < -133) ue = -133; /* subnormal spacing 2^-133 */
    double ulp = ldexp(1.0, ue);
    double q = floor(a / ulp);
    double rem = a - q * ulp;
    if (rem > 0.5 * ulp || (rem == 0.5 * ulp && fmod(q, 2.0) == 1.0)) q += 1.0;
    double r = q * ulp;
    if (r > 3.3895313892515355e38) return (uint16_t)(sign | 0x7f80); /* overflow to inf */
    float f = (float)r; /* exact */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7fff));
}

/* ------------------------------------------------------------------ */
/* e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;       */
/* no infinities; S.1111.111 is NaN; largest finite 448 (0x7E).       */
/* (FP8 formats, OCP 8-bit floating point specification, E4M3.)       */
/* ------------------------------------------------------------------ */

static double E4M3[256];
static int e4m3_ready = 0;

static void e4m3_init(void) {
    if (e4m3_ready) return;
    for (int c = 0; c < 256; ++c) {
        int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
        double v;
        if (e == 15 && m == 7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)m / 8.0, -6); /* subnormal: (m/8) * 2^(1-7) */
        else
            v = ldexp(1.0 + (double)m / 8.0, e - 7);
        E4M3[c] = s ? -v : v;
    }
    e4m3_ready = 1;
}

double oracle_e4m3_decode(uint8_t c) {
    e4m3_init();
    return E4M3[c];
}

/* Reference encoder: nearest finite value by scanning every non-negative
 * finite code, ties to the even code, |v| above 448 saturates to 448, the
 * sign is kept (so a negative value that rounds to zero gives 0x80). */
uint8_t oracle_e4m3_encode_scan(float v) {
    e4m3_init();
    if (isnan(v)) return 0x7f;
    double a = fabs((double)v);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        double d = fabs(E4M3[c] - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 0x80 : 0));
}

/* Same mapping, found by bisection over the 127 non-negative finite codes,
 * whose values increase with the code. */
uint8_t oracle_e4m3_encode(float v) {
    e4m3_init();
    if (isnan(v)) return 0x7f;
    double a = fabs((double)v);
    int c;
    if (a >= E4M3[0x7e]) {
        c = 0x7e;
    } else {
        int lo = 0, hi = 0x7e; /* E4M3[lo] <= a < E4M3[hi] */
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (E4M3[mid] <= a)
                lo = mid;
            else
                hi = mid;
        }
        double dl = a - E4M3[lo], dh = E4M3[hi] - a;
        if (dl < dh)
            c = lo;
        else if (dh < dl)
            c = hi;
        else
            c = (lo & 1) == 0 ? lo : hi;
    }
    return (uint8_t)(c | (signbit(v) ? 0x80 : 0));
}

/* ------------------------------------------------------------------ */
/* Quantisers                                                         */
/* ------------------------------------------------------------------ */

/* One group of n <= 128 fp32 values (the rest of the 128 are zero pad):
 * s = amax/448 (fp32), code = e4m3(v/s) (fp32 division). */
static float quant_group(const float* v, int n, uint8_t* q) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int i = 0; i < 128; ++i) q[i] = 0;
        return 1.0f;
    }
    float s = amax / 448.0f;
    for (int i = 0; i < n; ++i) {
        float t = v[i] / s;
        q[i] = oracle_e4m3_encode(t);
    }
    for (int i = n; i < 128; ++i) q[i] = 0;
    return s;
}

/* 1x128 per-token-group quantisation of one row of `cols` fp32 values into
 * `ceil(cols/128)*128` codes and one scale per group (x before the gate/up
 * GEMM, h before the down GEMM). */
void oracle_quant_row_1x128(const float* v, int cols, uint8_t* q, float* s) {
    int groups = (cols + 127) / 128;
    for (int g = 0; g < groups; ++g) {
        int n = cols - g * 128;
        if (n > 128) n = 128;
        s[g] = quant_group(v + (size_t)g * 128, n, q + (size_t)g * 128);
    }
}

/* same, rows of bf16 input */
void oracle_quant_rows_bf16(const uint16_t* x, int rows, int cols, uint8_t* q, float* s) {
    int cp = (cols + 127) / 128 * 128;
    float* tmp = (float*)malloc(sizeof(float) * (size_t)cols);
    for (int r = 0; r < rows; ++r) {
        for (int c = 0; c < cols; ++c) tmp[c] = (float)bf16_value(x[(size_t)r * cols + c]);
        oracle_quant_row_1x128(tmp, cols, q + (size_t)r * cp, s + (size_t)r * (cp / 128));
    }
    free(tmp);
}

/* same, rows of fp32 input (the requant step on its own) */
void oracle_quant_rows_f32(const float* x, int rows, int cols, uint8_t* q, float* s) {
    int cp = (cols + 127) / 128 * 128;
    for (int r = 0; r < rows; ++r)
        oracle_quant_row_1x128(x + (size_t)r * cols, cols, q + (size_t)r * cp, s + (size_t)r * (cp / 128));
}

/* 128x128 block quantisation of a [rows, cols] fp32 matrix into a zero-padded
 * [rows_p, cols_p] code matrix placed at row dst_row0 of a matrix with
 * cols_p columns, with block scales [rows_p/128, cols_p/128] placed at
 * block-row dst_row0/128.  Blocks are taken over the padded layout; zero pad
 * never raises amax.  (FP8 with 128x128 block scaling: "GPT-OSS on Day 0",
 * infrastructure decisions list.) */
static void quant_blocks(const float* w, int rows, int cols, int cols_p, uint8_t* q, float* s, int dst_row0) {
    int kb_n = cols_p / 128;
    int rb_n = (rows + 127) / 128;
    for (int rb = 0; rb < rb_n; ++rb) {
        for (int kb = 0; kb < kb_n; ++kb) {
            int r_end = rb * 128 + 128 < rows ? rb * 128 + 128 : rows;
            int c_end = kb * 128 + 128 < cols ? kb * 128 + 128 : cols;
            float amax = 0.0f;
            for (int r = rb * 128; r < r_end; ++r)
                for (int c = kb * 128; c < c_end; ++c) {
                    float a = fabsf(w[(size_t)r * cols + c]);
                    if (a > amax) amax = a;
                }
            float sc = amax == 0.0f ? 1.0f : amax / 448.0f;
            s[(size_t)(dst_row0 / 128 + rb) * kb_n + kb] = sc;
            for (int r = rb * 128; r < rb * 128 + 128; ++r)
                for (int c = kb * 128; c < kb * 128 + 128; ++c) {
                    uint8_t code = 0;
                    if (amax != 0.0f && r < rows && c < cols) code = oracle_e4m3_encode(w[(size_t)r * cols + c] / sc);
                    q[(size_t)(dst_row0 + r) * cols_p + c] = code;
                }
        }
    }
}

/* w13 master [n_exp, 2I, H] (gate rows then up rows) -> codes [n_exp, 2Ip, Hp],
 * scales [n_exp, 2Ip/128, Hp/128]; gate goes to rows [0,I), up to [Ip, Ip+I). */
void oracle_pack_w13(const float* w13, int H, int I, int n_exp, uint8_t* q, float* s) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    for (int e = 0; e < n_exp; ++e) {
        const float* we = w13 + (size_t)e * 2 * I * H;
        uint8_t* qe = q + (size_t)e * 2 * Ip * Hp;
        float* se = s + (size_t)e * (2 * Ip / 128) * (Hp / 128);
        quant_blocks(we, I, H, Hp, qe, se, 0);
        quant_blocks(we + (size_t)I * H, I, H, Hp, qe, se, Ip);
    }
}

/* w2 master [n_exp, H, I] -> codes [n_exp, Hp, Ip], scales [n_exp, Hp/128, Ip/128] */
void oracle_pack_w2(const float* w2, int H, int I, int n_exp, uint8_t* q, float* s) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    for (int e = 0; e < n_exp; ++e)
        quant_blocks(w2 + (size_t)e * H * I, H, I, Ip, q + (size_t)e * Hp * Ip, s + (size_t)e * (Hp / 128) * (Ip / 128),
                     0);
}

/* ------------------------------------------------------------------ */
/* Router: logits, top-k, softmax over the selected k                 */
/* ("GPT-OSS on Day 0": MoE MLP bullets -- softmax after top-k; the   */
/* routing paragraph -- softmax only over the selected experts, expert */
/* weights in bfloat16.)                                              */
/* ------------------------------------------------------------------ */

/* One token.  logits[e] = sum_h x[h]*Wr[e,h] + br[e] in fp64 over the bf16
 * values.  Selects the k largest (ties -> lower e), stores them in ascending
 * expert order, and the softmax weights over those k logits (fp64 -> fp32 ->
 * bf16).  margin = (k-th largest) - ((k+1)-th largest), +inf when k == E. */
static void route_token(const uint16_t* x, const uint16_t* rw, const uint16_t* rb, int H, int E, int k, int32_t* idx,
                        float* w_f32, uint16_t* w_bf16, double* logits, double* margin) {
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h) acc += bf16_value(x[h]) * bf16_value(rw[(size_t)e * H + h]);
        logits[e] = acc + bf16_value(rb[e]);
    }
    char* taken = (char*)calloc((size_t)E, 1);
    double kth = 0.0;
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e)
            if (!taken[e] && (best < 0 || logits[e] > logits[best])) best = e;
        taken[best] = 1;
        kth = logits[best];
    }
    double next = -INFINITY;
    for (int e = 0; e < E; ++e)
        if (!taken[e] && logits[e] > next) next = logits[e];
    if (margin) *margin = (k < E) ? kth - next : INFINITY;
    /* ascending expert order */
    int n = 0;
    for (int e = 0; e < E; ++e)
        if (taken[e]) idx[n++] = e;
    free(taken);
    double m = -INFINITY;
    for (int j = 0; j < k; ++j)
        if (logits[idx[j]] > m) m = logits[idx[j]];
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += exp(logits[idx[j]] - m);
    for (int j = 0; j < k; ++j) {
        double w = exp(logits[idx[j]] - m) / z;
        w_f32[j] = (float)w;
        w_bf16[j] = oracle_bf16_from_f32(w_f32[j]);
    }
}

void oracle_router(const uint16_t* x, const uint16_t* rw, const uint16_t* rb, int T, int H, int E, int k,
                   int32_t* idx, float* w_f32, uint16_t* w_bf16, double* logits_out, double* margin_out) {
    double* logits = (double*)malloc(sizeof(double) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        route_token(x + (size_t)t * H, rw, rb, H, E, k, idx + (size_t)t * k, w_f32 + (size_t)t * k,
                    w_bf16 + (size_t)t * k, logits, margin_out ? margin_out + t : NULL);
        if (logits_out) memcpy(logits_out + (size_t)t * E, logits, sizeof(double) * (size_t)E);
    }
    free(logits);
}

/* ------------------------------------------------------------------ */
/* Grouping tokens by expert (the dispatch side of dispatch/combine): */
/* counting sort of the (token, slot) pairs by (expert, token).       */
/* ------------------------------------------------------------------ */
void oracle_permute(const int32_t* idx, int T, int E, int k, int32_t* count, int32_t* offset, int32_t* perm,
                    int32_t* inv) {
    for (int e = 0; e < E; ++e) count[e] = 0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) count[idx[(size_t)t * k + j]]++;
    offset[0] = 0;
    for (int e = 0; e < E; ++e) offset[e + 1] = offset[e] + count[e];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = idx[(size_t)t * k + j];
            int r = offset[e] + fill[e]++;
            perm[r] = t * k + j;
            inv[(size_t)t * k + j] = r;
        }
    free(fill);
}

/* ------------------------------------------------------------------ */
/* Expert GEMMs with 128x128 block-scaled FP8 weights                 */
/* ------------------------------------------------------------------ */

/* out[n] for n in [0, N): sum over K-blocks kb of (sa[kb] * sw[n/128, kb]) *
 * sum_{i in kb} dec(a[i]) * dec(w[n, i]), in fp64; a is one row of Kp codes,
 * w is [Np, Kp] codes, sw is [Np/128, Kp/128]. */
static double block_scaled_dot(const uint8_t* a, const float* sa, const uint8_t* w, const float* sw, int n, int Kp) {
    int kbn = Kp / 128;
    double acc = 0.0;
    for (int kb = 0; kb < kbn; ++kb) {
        double part = 0.0;
        for (int i = kb * 128; i < kb * 128 + 128; ++i) part += E4M3[a[i]] * E4M3[w[(size_t)n * Kp + i]];
        acc += ((double)sa[kb] * (double)sw[(size_t)(n / 128) * kbn + kb]) * part;
    }
    return acc;
}

/* One (token, expert) pair: h = silu(g)*u of the gate/up GEMM with b13
 * ("experts have biases"; SwiGLU activation), requantised 1x128, then
 * y = down GEMM + b2.  xq/sx: the token's quantised row [Hp], [Hp/128].
 * Writes hq [Ip], sh [Ip/128], y [H] (fp64). */
static void expert_ffn(const uint8_t* xq, const float* sx, const uint8_t* w13e, const float* s13e,
                       const uint16_t* b13e, const uint8_t* w2e, const float* s2e, const uint16_t* b2e, int H, int I,
                       uint8_t* hq, float* sh, double* y) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    float* h = (float*)malloc(sizeof(float) * (size_t)I);
    for (int n = 0; n < I; ++n) {
        double g = (double)bf16_value(b13e[n]) + block_scaled_dot(xq, sx, w13e, s13e, n, Hp);
        double u = (double)bf16_value(b13e[I + n]) + block_scaled_dot(xq, sx, w13e, s13e, Ip + n, Hp);
        double silu = g / (1.0 + exp(-g));
        h[n] = (float)(silu * u);
    }
    oracle_quant_row_1x128(h, I, hq, sh);
    free(h);
    for (int n = 0; n < H; ++n) y[n] = (double)bf16_value(b2e[n]) + block_scaled_dot(hq, sh, w2e, s2e, n, Ip);
}

/* Full layer for a list of tokens (all T when tokens == NULL).
 * out_rows [ntok, H] bf16 bits.  Optional: hq_rows [ntok*k, Ip],
 * sh_rows [ntok*k, Ip/128], y_rows [ntok*k, H] (fp64 expert outputs),
 * idx_rows [ntok*k].  The k expert outputs are combined as the weighted sum
 * p_j = w_j(bf16) * y_j, out = bf16(sum_j p_j) ("Combine performs the
 * weighted accumulation"). */
void oracle_forward(const uint16_t* x, const uint16_t* rw, const uint16_t* rb, const uint8_t* w13, const float* s13,
                    const uint16_t* b13, const uint8_t* w2, const float* s2, const uint16_t* b2, int T, int H, int I,
                    int E, int k, const int32_t* tokens, int ntok, uint16_t* out_rows, uint8_t* hq_rows,
                    float* sh_rows, double* y_rows, int32_t* idx_rows) {
    e4m3_init();
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    if (!tokens) ntok = T;
    double* logits = (double*)malloc(sizeof(double) * (size_t)E);
    uint8_t* xq = (uint8_t*)malloc((size_t)Hp);
    float* sx = (float*)malloc(sizeof(float) * (size_t)(Hp / 128));
    uint8_t* hq = (uint8_t*)malloc((size_t)Ip);
    float* sh = (float*)malloc(sizeof(float) * (size_t)(Ip / 128));
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    int32_t idx[64];
    float wf[64];
    uint16_t wb[64];
    for (int i = 0; i < ntok; ++i) {
        int t = tokens ? tokens[i] : i;
        const uint16_t* xt = x + (size_t)t * H;
        route_token(xt, rw, rb, H, E, k, idx, wf, wb, logits, NULL);
        oracle_quant_rows_bf16(xt, 1, H, xq, sx);
        for (int n = 0; n < H; ++n) acc[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = idx[j];
            expert_ffn(xq, sx, w13 + (size_t)e * 2 * Ip * Hp, s13 + (size_t)e * (2 * Ip / 128) * (Hp / 128),
                       b13 + (size_t)e * 2 * I, w2 + (size_t)e * Hp * Ip, s2 + (size_t)e * (Hp / 128) * (Ip / 128),
                       b2 + (size_t)e * H, H, I, hq, sh, y);
            double wj = bf16_value(wb[j]);
            for (int n = 0; n < H; ++n) acc[n] += wj * y[n];
            size_t row = (size_t)i * k + j;
            if (hq_rows) memcpy(hq_rows + row * Ip, hq, (size_t)Ip);
            if (sh_rows) memcpy(sh_rows + row * (Ip / 128), sh, sizeof(float) * (size_t)(Ip / 128));
            if (y_rows) memcpy(y_rows + row * H, y, sizeof(double) * (size_t)H);
            if (idx_rows) idx_rows[row] = e;
        }
        for (int n = 0; n < H; ++n) out_rows[(size_t)i * H + n] = oracle_bf16_from_f64(acc[n]);
    }
    free(logits);
    free(xq);
    free(sx);
    free(hq);
    free(sh);
    free(y);
    free(acc);
}

/* ------------------------------------------------------------------ */
/* MXFP8 variant                                                      */
/* ------------------------------------------------------------------ */
/* "Hosting Qwen on Blackwell" (section "Quantization"): on Blackwell the
 * throughput case for FP8 is microscaling, one power-of-two scale per 32
 * consecutive values.  The scale is the one the OCP Microscaling Formats
 * (MX) specification v1.0 (section 6.3) defines: for a group of 32 values,
 * X = floor(log2(max |v|)) - 8 (8 = the exponent of e4m3's largest normal,
 * 448 = 1.75 * 2^8), kept as the UE8M0 byte X + 127; the codes are
 * e4m3(v / 2^X) -- nearest, ties to even, saturating to +-448 (values of the
 * top binade above 448 saturate, as the specification allows).  Readings
 * where that is silent (also in the design notes): an all-zero group gets the
 * byte 0 (2^-127) and +0 codes; X is clamped to [-127, 127]; the layer is the
 * same pipeline as the 128x128 variant with every quantiser replaced by this
 * one (x along H, h along I, weight rows along K), padding to multiples of
 * 128 as there. */
static uint8_t mx_group(const float* v, int n, uint8_t* q) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    for (int i = 0; i < 32; ++i) q[i] = 0;
    if (amax == 0.0f) return 0;
    int e;
    frexp((double)amax, &e); /* amax = f * 2^e, f in [0.5, 1): floor(log2(amax)) = e - 1 */
    int X = e - 1 - 8;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    for (int i = 0; i < n; ++i) q[i] = oracle_e4m3_encode((float)ldexp((double)v[i], -X));
    return (uint8_t)(X + 127);
}

/* MX quantisation of `rows` rows of `cols` fp32 values: codes [rows, Cp] and
 * scale bytes [rows, Cp/32], Cp = cols padded to a multiple of 128. */
void oracle_mx_quant_rows_f32(const float* x, int rows, int cols, uint8_t* q, uint8_t* s) {
    int Cp = (cols + 127) / 128 * 128;
    for (int r = 0; r < rows; ++r)
        for (int g = 0; g < Cp / 32; ++g) {
            int c0 = g * 32;
            int n = cols - c0 < 32 ? (cols - c0 > 0 ? cols - c0 : 0) : 32;
            s[(size_t)r * (Cp / 32) + g] = mx_group(x + (size_t)r * cols + c0, n, q + (size_t)r * Cp + c0);
        }
}

void oracle_mx_quant_rows_bf16(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* s) {
    float* f = (float*)malloc(sizeof(float) * (size_t)rows * cols);
    for (size_t i = 0; i < (size_t)rows * cols; ++i) f[i] = (float)bf16_value(x[i]);
    oracle_mx_quant_rows_f32(f, rows, cols, q, s);
    free(f);
}

/* Weights: every output row quantised along K.  w13 [n_exp, 2I, H] ->
 * q [n_exp, 2Ip, Hp] (gate rows [0,I), up rows [Ip, Ip+I), pad rows 0),
 * s [n_exp, 2Ip, Hp/32]; w2 [n_exp, H, I] -> q [n_exp, Hp, Ip],
 * s [n_exp, Hp, Ip/32].  Pad rows have the byte 0 and codes 0. */
static void mx_pack(const float* w, int rows, int cols, int rows_p, int cols_p, const int* row_map, uint8_t* q,
                    uint8_t* s) {
    memset(q, 0, (size_t)rows_p * cols_p);
    memset(s, 0, (size_t)rows_p * (cols_p / 32));
    uint8_t* qr = (uint8_t*)malloc((size_t)cols_p);
    uint8_t* sr = (uint8_t*)malloc((size_t)cols_p / 32);
    for (int r = 0; r < rows; ++r) {
        oracle_mx_quant_rows_f32(w + (size_t)r * cols, 1, cols, qr, sr);
        int d = row_map ? row_map[r] : r;
        memcpy(q + (size_t)d * cols_p, qr, (size_t)cols_p);
        memcpy(s + (size_t)d * (cols_p / 32), sr, (size_t)cols_p / 32);
    }
    free(qr);
    free(sr);
}

void oracle_mx_pack_w13(const float* w13, int H, int I, int n_exp, uint8_t* q, uint8_t* s) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    int* map = (int*)malloc(sizeof(int) * 2 * (size_t)I);
    for (int r = 0; r < I; ++r) {
        map[r] = r;
        map[I + r] = Ip + r;
    }
    for (int e = 0; e < n_exp; ++e)
        mx_pack(w13 + (size_t)e * 2 * I * H, 2 * I, H, 2 * Ip, Hp, map, q + (size_t)e * 2 * Ip * Hp,
                s + (size_t)e * 2 * Ip * (Hp / 32));
    free(map);
}

void oracle_mx_pack_w2(const float* w2, int H, int I, int n_exp, uint8_t* q, uint8_t* s) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    for (int e = 0; e < n_exp; ++e)
        mx_pack(w2 + (size_t)e * H * I, H, I, Hp, Ip, NULL, q + (size_t)e * Hp * Ip, s + (size_t)e * Hp * (Ip / 32));
}

/* sum over 32-groups g of 2^(sa[g]-127) * 2^(sw[n,g]-127) * sum_{i in g}
 * dec(a[i]) * dec(w[n,i]), in fp64 (exact: e4m3 products and their sums over
 * 32 fit in fp64, the scales are powers of two). */
static double mx_dot(const uint8_t* a, const uint8_t* sa, const uint8_t* w, const uint8_t* sw, int n, int Kp,
                     const double* wtab) {
    int G = Kp / 32;
    double acc = 0.0;
    for (int g = 0; g < G; ++g) {
        double part = 0.0;
        for (int i = g * 32; i < g * 32 + 32; ++i) part += E4M3[a[i]] * wtab[w[(size_t)n * Kp + i]];
        acc += ldexp(part, ((int)sa[g] - 127) + ((int)sw[(size_t)n * G + g] - 127));
    }
    return acc;
}

/* wtab: decode table of the weight codes (E4M3 for MXFP8 weights, E2M1 for
 * MXFP4 weights); activations are MXFP8 either way. */
static void mx_expert_ffn(const uint8_t* xq, const uint8_t* sx, const uint8_t* w13e, const uint8_t* s13e,
                          const uint16_t* b13e, const uint8_t* w2e, const uint8_t* s2e, const uint16_t* b2e, int H,
                          int I, uint8_t* hq, uint8_t* sh, double* y, const double* wtab) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    float* h = (float*)malloc(sizeof(float) * (size_t)I);
    for (int n = 0; n < I; ++n) {
        double g = (double)bf16_value(b13e[n]) + mx_dot(xq, sx, w13e, s13e, n, Hp, wtab);
        double u = (double)bf16_value(b13e[I + n]) + mx_dot(xq, sx, w13e, s13e, Ip + n, Hp, wtab);
        double silu = g / (1.0 + exp(-g));
        h[n] = (float)(silu * u);
    }
    oracle_mx_quant_rows_f32(h, 1, I, hq, sh);
    free(h);
    for (int n = 0; n < H; ++n) y[n] = (double)bf16_value(b2e[n]) + mx_dot(hq, sh, w2e, s2e, n, Ip, wtab);
}

/* The layer with MXFP8 quantisation; arguments as oracle_forward, with the
 * scale arrays in UE8M0 bytes (s13 [E, 2Ip, Hp/32], s2 [E, Hp, Ip/32]) and
 * sh_rows [ntok*k, Ip/32]. */
static void mx_forward_impl(const uint16_t* x, const uint16_t* rw, const uint16_t* rb, const uint8_t* w13,
                            const uint8_t* s13, const uint16_t* b13, const uint8_t* w2, const uint8_t* s2,
                            const uint16_t* b2, int T, int H, int I, int E, int k, const int32_t* tokens, int ntok,
                            uint16_t* out_rows, uint8_t* hq_rows, uint8_t* sh_rows, double* y_rows, int32_t* idx_rows,
                            const double* wtab) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    if (!tokens) ntok = T;
    double* logits = (double*)malloc(sizeof(double) * (size_t)E);
    uint8_t* xq = (uint8_t*)malloc((size_t)Hp);
    uint8_t* sx = (uint8_t*)malloc((size_t)Hp / 32);
    uint8_t* hq = (uint8_t*)malloc((size_t)Ip);
    uint8_t* sh = (uint8_t*)malloc((size_t)Ip / 32);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    int32_t idx[64];
    float wf[64];
    uint16_t wb[64];
    for (int i = 0; i < ntok; ++i) {
        int t = tokens ? tokens[i] : i;
        const uint16_t* xt = x + (size_t)t * H;
        route_token(xt, rw, rb, H, E, k, idx, wf, wb, logits, NULL);
        oracle_mx_quant_rows_bf16(xt, 1, H, xq, sx);
        for (int n = 0; n < H; ++n) acc[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = idx[j];
            mx_expert_ffn(xq, sx, w13 + (size_t)e * 2 * Ip * Hp, s13 + (size_t)e * 2 * Ip * (Hp / 32),
                          b13 + (size_t)e * 2 * I, w2 + (size_t)e * Hp * Ip, s2 + (size_t)e * Hp * (Ip / 32),
                          b2 + (size_t)e * H, H, I, hq, sh, y, wtab);
            double wj = bf16_value(wb[j]);
            for (int n = 0; n < H; ++n) acc[n] += wj * y[n];
            size_t row = (size_t)i * k + j;
            if (hq_rows) memcpy(hq_rows + row * Ip, hq, (size_t)Ip);
            if (sh_rows) memcpy(sh_rows + row * (Ip / 32), sh, (size_t)Ip / 32);
            if (y_rows) memcpy(y_rows + row * H, y, sizeof(double) * (size_t)H);
            if (idx_rows) idx_rows[row] = e;
        }
        for (int n = 0; n < H; ++n) out_rows[(size_t)i * H + n] = oracle_bf16_from_f64(acc[n]);
    }
    free(logits);
    free(xq);
    free(sx);
    free(hq);
    free(sh);
    free(y);
    free(acc);
}

void oracle_mx_forward(const uint16_t* x, const uint16_t* rw, const uint16_t* rb, const uint8_t* w13,
                       const uint8_t* s13, const uint16_t* b13, const uint8_t* w2, const uint8_t* s2,
                       const uint16_t* b2, int T, int H, int I, int E, int k, const int32_t* tokens, int ntok,
                       uint16_t* out_rows, uint8_t* hq_rows, uint8_t* sh_rows, double* y_rows, int32_t* idx_rows) {
    e4m3_init();
    mx_forward_impl(x, rw, rb, w13, s13, b13, w2, s2, b2, T, H, I, E, k, tokens, ntok, out_rows, hq_rows, sh_rows,
                    y_rows, idx_rows, E4M3);
}

/* ------------------------------------------------------------------ */
/* MXFP4 weights                                                      */
/* ------------------------------------------------------------------ */
/* "GPT-OSS on Day 0" (opening section): the open-weight models ship with
 * MXFP4 quantisation, and the FP4 tensor cores that run it natively are new
 * with Blackwell.  OCP Microscaling Formats (MX) v1.0: the element format is
 * FP4 E2M1 (section 5.3.3: 1 sign bit, 2 exponent bits with bias 1, 1
 * mantissa bit, no infinities or NaN; exponent field 0 is subnormal, m * 0.5;
 * otherwise (1 + m/2) * 2^(e-1): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), the
 * block is 32 values with one UE8M0 scale, and the shared exponent is
 * X = floor(log2(amax)) - 2 (section 6.3; 2 = the exponent of E2M1's largest
 * normal).  Codes: e2m1(v / 2^X), nearest, ties to the even code, saturating
 * to +-6 (values of the top binade above 6).  The readings of the MXFP8
 * section carry over (all-zero group: byte 0 and +0 codes; X clamped to
 * [-127, 127]).  The layer: weights in MXFP4 along K, x and h in MXFP8 --
 * FP4 codes with FP8 activations.  Codes are kept one per byte here (the low
 * 4 bits: sign in bit 3). */
static double E2M1[16];
static int e2m1_ready = 0;

static void e2m1_init(void) {
    if (e2m1_ready) return;
    for (int c = 0; c < 16; ++c) {
        int sgn = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
        double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
        E2M1[c] = sgn ? -v : v;
    }
    e2m1_ready = 1;
}

double oracle_e2m1_decode(uint8_t c) {
    e2m1_init();
    return E2M1[c & 15];
}

/* Nearest E2M1 code of an fp32 value, ties to the even code (even mantissa
 * bit), saturating to +-6; the sign is kept for values that round to 0. */
uint8_t oracle_e2m1_encode(float v) {
    e2m1_init();
    double a = fabs((double)v);
    uint8_t sgn = signbit(v) ? 8 : 0;
    int c;
    if (a >= E2M1[7]) {
        c = 7;
    } else {
        int lo = 0, hi = 7; /* E2M1[lo] <= a < E2M1[hi] */
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (E2M1[mid] <= a)
                lo = mid;
            else
                hi = mid;
        }
        double dl = a - E2M1[lo], dh = E2M1[hi] - a;
        c = dl < dh ? lo : (dh < dl ? hi : ((lo & 1) == 0 ? lo : hi));
    }
    return (uint8_t)(sgn | c);
}

static uint8_t mx4_group(const float* v, int n, uint8_t* q) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    for (int i = 0; i < 32; ++i) q[i] = 0;
    if (amax == 0.0f) return 0;
    int e;
    frexp((double)amax, &e); /* floor(log2(amax)) = e - 1 */
    int X = e - 1 - 2;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    for (int i = 0; i < n; ++i) q[i] = oracle_e2m1_encode((float)ldexp((double)v[i], -X));
    return (uint8_t)(X + 127);
}

/* MXFP4 quantisation of rows: codes [rows, Cp] (one per byte), scale bytes
 * [rows, Cp/32], Cp = cols padded to a multiple of 128. */
void oracle_mx4_quant_rows_f32(const float* x, int rows, int cols, uint8_t* q, uint8_t* s) {
    int Cp = (cols + 127) / 128 * 128;
    for (int r = 0; r < rows; ++r)
        for (int g = 0; g < Cp / 32; ++g) {
            int c0 = g * 32;
            int n = cols - c0 < 32 ? (cols - c0 > 0 ? cols - c0 : 0) : 32;
            s[(size_t)r * (Cp / 32) + g] = mx4_group(x + (size_t)r * cols + c0, n, q + (size_t)r * Cp + c0);
        }
}

static void mx4_pack(const float* w, int rows, int cols, int rows_p, int cols_p, const int* row_map, uint8_t* q,
                     uint8_t* s) {
    memset(q, 0, (size_t)rows_p * cols_p);
    memset(s, 0, (size_t)rows_p * (cols_p / 32));
    for (int r = 0; r < rows; ++r) {
        int d = row_map ? row_map[r] : r;
        oracle_mx4_quant_rows_f32(w + (size_t)r * cols, 1, cols, q + (size_t)d * cols_p, s + (size_t)d * (cols_p / 32));
    }
}

/* Weights in MXFP4: w13 [n_exp, 2I, H] -> codes [n_exp, 2Ip, Hp], scale
 * bytes [n_exp, 2Ip, Hp/32] (gate rows [0,I), up rows [Ip, Ip+I)); w2
 * [n_exp, H, I] -> codes [n_exp, Hp, Ip], bytes [n_exp, Hp, Ip/32]. */
void oracle_mx4_pack_w13(const float* w13, int H, int I, int n_exp, uint8_t* q, uint8_t* s) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    int* map = (int*)malloc(sizeof(int) * 2 * (size_t)I);
    for (int r = 0; r < I; ++r) {
        map[r] = r;
        map[I + r] = Ip + r;
    }
    for (int e = 0; e < n_exp; ++e)
        mx4_pack(w13 + (size_t)e * 2 * I * H, 2 * I, H, 2 * Ip, Hp, map, q + (size_t)e * 2 * Ip * Hp,
                 s + (size_t)e * 2 * Ip * (Hp / 32));
    free(map);
}

void oracle_mx4_pack_w2(const float* w2, int H, int I, int n_exp, uint8_t* q, uint8_t* s) {
    int Hp = (H + 127) / 128 * 128, Ip = (I + 127) / 128 * 128;
    for (int e = 0; e < n_exp; ++e)
        mx4_pack(w2 + (size_t)e * H * I, H, I, Hp, Ip, NULL, q + (size_t)e * Hp * Ip, s + (size_t)e * Hp * (Ip / 32));
}

/* The layer with MXFP4 weights (codes one per byte) and MXFP8 activations;
 * arguments as oracle_mx_forward. */
void oracle_mx4_forward(const uint16_t* x, const uint16_t* rw, const uint16_t* rb, const uint8_t* w13,
                        const uint8_t* s13, const uint16_t* b13, const uint8_t* w2, const uint8_t* s2,
                        const uint16_t* b2, int T, int H, int I, int E, int k, const int32_t* tokens, int ntok,
                        uint16_t* out_rows, uint8_t* hq_rows, uint8_t* sh_rows, double* y_rows, int32_t* idx_rows) {
    e4m3_init();
    e2m1_init();
    mx_forward_impl(x, rw, rb, w13, s13, b13, w2, s2, b2, T, H, I, E, k, tokens, ntok, out_rows, hq_rows, sh_rows,
                    y_rows, idx_rows, E2M1);
}

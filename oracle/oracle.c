/*
 * oracle.c -- plain, slow, fp64 CPU reference of the routed-MoE FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA path of the package, and the
 * package never calls it.
 *
 * What it computes ("Systems engineering playbook: Qwen 3.5 MoE on Ironwood
 * TPU"; the Vietnamese translation of the report, section 1.3 "Sparse
 * Mixture-of-Experts", and the English page, sections "The Architectural
 * Constraints That Break Naive Sharding" and "Fusing Three Collectives Into
 * Two"):
 *   - a router gate projects each token to one logit per expert,
 *   - the top 10 experts are chosen through a softmax distribution and their
 *     weights renormalised over the chosen set,
 *   - each chosen expert (a SwiGLU FFN of intermediate 1024) runs on the
 *     token, and an always-on shared expert is added,
 *   - expert indices and weights travel as one 32-bit blob (two [T,k] planes).
 * The pages lose the output equation itself; the reading used here is
 *   out[t] = shared(x_t) + sum_j w[t,j] * expert_{idx[t,j]}(x_t),
 * with the shared expert unweighted.
 *
 * Everything is computed in double from the exact input values; bf16, fp32
 * and E4M3 inputs convert to double without loss through this file's own
 * codecs.  No blocking, fusion or reordering beyond the definitions.
 *
 * Parity pins (tests/test_oracle_pins.py): codecs against an exhaustive
 * table and torch casts; top-k against a brute-force stable sort with
 * planted ties; weights sum to one and top_k = E reproduces the dense softmax
 * mixture; E = 1, k = 1 reproduces a dense SwiGLU FFN computed with numpy;
 * identity experts make permute-then-unpermute the identity; counts sum to
 * T*k and the permutation is a bijection; token-order equivariance and
 * expert relabelling invariance; the 128x128 weight-block and the per-row
 * 128-column activation quantisers against torch's E4M3 cast, and the FP8
 * layer with one expert against numpy over that cast; the whole layer against closed forms computed
 * with numpy and scipy: top_k = E is the dense softmax mixture, and top_k < E with every expert
 * outside a random chosen set biased 1000 below it (zero softmax mass in fp64) is that same dense
 * mixture.  The pages print no worked value of the layer; these closed forms pin it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_EXPORT __attribute__((visibility("default")))

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

/* ------------------------------------------------------------------ codecs */

/* bf16 is the top half of an IEEE binary32. */
ORC_EXPORT double orc_bf16_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* binary32 -> bf16, round to nearest, ties to even; NaN stays a quiet NaN. */
ORC_EXPORT uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16, rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

/* OCP FP8 E4M3 ("fn" variant): bias 7, no infinities, S.1111.111 is NaN,
 * largest finite 448, subnormal quantum 2^-9. */
ORC_EXPORT double orc_e4m3_to_f64(uint8_t q) {
    int s = q >> 7, e = (q >> 3) & 15, m = q & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* binary32 -> E4M3, round to nearest even, saturating to +-448 (finite in).
 * The magnitude is scaled to an integer count of the quantum of its binade,
 * rounded, and the code is (binade << 3) + mantissa; a carry out of the
 * mantissa lands on the next binade's first code, so codes stay contiguous. */
ORC_EXPORT uint8_t orc_f32_to_e4m3(float f) {
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    if (isnan(f)) return 0x7f;
    double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7e;
    int code;
    if (a < ldexp(1.0, -6)) {                  /* subnormal range */
        double n = a / ldexp(1.0, -9);         /* exact: power-of-two scale */
        double fl = floor(n), fr = n - fl;
        long m = (long)fl;
        if (fr > 0.5 || (fr == 0.5 && (m & 1))) m += 1;
        code = (int)m;                         /* m == 8 is the first normal */
    } else {
        int ex;
        double fr0 = frexp(a, &ex);            /* a = fr0 * 2^ex, fr0 in [0.5,1) */
        int E = ex - 1;                        /* a in [2^E, 2^(E+1)) */
        double n = ldexp(a, 3 - E);            /* in [8, 16) */
        (void)fr0;
        double fl = floor(n), fr = n - fl;
        long m = (long)fl;
        if (fr > 0.5 || (fr == 0.5 && (m & 1))) m += 1;
        code = ((E + 7) << 3) + (int)(m - 8);
    }
    if (code > 0x7e) code = 0x7e;
    return (uint8_t)(sign | code);
}

ORC_EXPORT void orc_e4m3_encode_array(int64_t n, const float* in, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(in[i]);
}
ORC_EXPORT void orc_bf16_encode_array(int64_t n, const float* in, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}

static inline double load_elem(int dt, const void* p, int64_t i) {
    if (dt == ORC_F32) return (double)((const float*)p)[i];
    if (dt == ORC_BF16) return orc_bf16_to_f64(((const uint16_t*)p)[i]);
    return orc_e4m3_to_f64(((const uint8_t*)p)[i]);
}

/* ----------------------------------------------------- block quantisation */

/* E4M3 with one fp32 scale per br x bc block of a row-major [rows, cols]
 * matrix: s = amax / 448 (s = 1 when the block is all zero), and each element
 * becomes E4M3(fp32(w * fp32(448 / amax))).  The value a code stands for is
 * code * s.  Weights use 128 x 128 blocks; activations use 1 x 128 (one scale
 * per token per 128-column group).  s is laid out [rows/br, cols/bc]. */
ORC_EXPORT void orc_quant_blocks(int64_t rows, int64_t cols, int64_t br, int64_t bc,
                                 const float* w, uint8_t* q, float* s) {
    int64_t nbr = rows / br, nbc = cols / bc;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nbr * nbc; ++b) {
        int64_t r0 = (b / nbc) * br, c0 = (b % nbc) * bc;
        float amax = 0.0f;
        for (int64_t r = r0; r < r0 + br; ++r)
            for (int64_t c = c0; c < c0 + bc; ++c) {
                float a = fabsf(w[r * cols + c]);
                if (a > amax) amax = a;
            }
        volatile float scale = amax / 448.0f;
        volatile float inv = 448.0f / amax;
        if (amax == 0.0f) { scale = 1.0f; inv = 1.0f; }
        s[b] = scale;
        for (int64_t r = r0; r < r0 + br; ++r)
            for (int64_t c = c0; c < c0 + bc; ++c) {
                volatile float p = w[r * cols + c] * inv;
                q[r * cols + c] = orc_f32_to_e4m3(p);
            }
    }
}

/* One row of activations through the 1 x 128 quantiser, returned as the
 * doubles the codes stand for (code * scale). */
static void quant_row_128(int64_t n, const float* v, double* deq) {
    for (int64_t c0 = 0; c0 < n; c0 += 128) {
        float amax = 0.0f;
        for (int64_t c = c0; c < c0 + 128; ++c) {
            float a = fabsf(v[c]);
            if (a > amax) amax = a;
        }
        volatile float scale = amax / 448.0f;
        volatile float inv = 448.0f / amax;
        if (amax == 0.0f) { scale = 1.0f; inv = 1.0f; }
        for (int64_t c = c0; c < c0 + 128; ++c) {
            volatile float p = v[c] * inv;
            deq[c] = orc_e4m3_to_f64(orc_f32_to_e4m3(p)) * (double)scale;
        }
    }
}

/* Rows of activations through quant_row_128, one row at a time (exported so
 * that the tests can pin the quantiser itself). */
ORC_EXPORT void orc_quant_rows_128(int64_t rows, int64_t cols, const float* v, double* deq) {
    for (int64_t r = 0; r < rows; ++r) quant_row_128(cols, v + r * cols, deq + r * cols);
}

/* ----------------------------------------------------------------- router */

/* z[t,e] = sum_d x[t,d] * w_r[e,d] + b[e], in double. */
ORC_EXPORT void orc_logits(int64_t T, int32_t D, int32_t E, int32_t x_dt, const void* x,
                           int32_t w_dt, const void* w_r, const float* bias, double* z) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int32_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int32_t d = 0; d < D; ++d)
                acc += load_elem(x_dt, x, t * D + d) * load_elem(w_dt, w_r, (int64_t)e * D + d);
            z[t * E + e] = acc + (bias ? (double)bias[e] : 0.0);
        }
}

/* Top-k by logit, largest first; of two equal logits the lower expert index
 * is taken first.  Picking by logit is picking by softmax probability (the
 * softmax is monotone) without the ties that rounding exp could create.
 * Weights: softmax restricted to the chosen set, which equals the full
 * softmax renormalised over the chosen set (the full denominator cancels):
 *   w_j = exp(z_j - z_max) / sum_{j' chosen} exp(z_j' - z_max). */
ORC_EXPORT void orc_topk(int64_t T, int32_t E, int32_t k, const double* z, int32_t* idx, double* w) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* zt = z + t * E;
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || zt[e] > zt[best])) best = e;
            taken[best] = 1;
            idx[t * k + j] = best;
        }
        free(taken);
        double zmax = zt[idx[t * k]], den = 0.0;
        for (int32_t j = 0; j < k; ++j) den += exp(zt[idx[t * k + j]] - zmax);
        for (int32_t j = 0; j < k; ++j) w[t * k + j] = exp(zt[idx[t * k + j]] - zmax) / den;
    }
}

/* ------------------------------------------------------------ permutation */

/* Expert-contiguous layout as a stable counting sort of the (t, j) pairs in
 * row-major [T, k] order:
 *   counts[e]  = number of pairs routed to e (e < E); counts[E] = T (shared)
 *   offsets    = exclusive prefix sum of counts, offsets[E] = T*k,
 *                offsets[E+1] = T*k + T
 *   p(t, j)    = offsets[e] + number of earlier pairs also routed to e
 *   inv[t*k+j] = p(t, j), src_tok[p] = t; the shared group holds every token
 *                in order at rows T*k .. T*k+T-1. */
ORC_EXPORT void orc_permute(int64_t T, int32_t E, int32_t k, const int32_t* idx, int32_t* counts,
                            int32_t* offsets, int32_t* inv, int32_t* src_tok) {
    for (int32_t e = 0; e <= E; ++e) counts[e] = 0;
    for (int64_t a = 0; a < T * k; ++a) counts[idx[a]] += 1;
    counts[E] = (int32_t)T;
    offsets[0] = 0;
    for (int32_t e = 0; e <= E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    for (int32_t e = 0; e <= E; ++e) cursor[e] = offsets[e];
    for (int64_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < k; ++j) {
            int32_t p = cursor[idx[t * k + j]]++;
            inv[t * k + j] = p;
            src_tok[p] = (int32_t)t;
        }
    for (int64_t t = 0; t < T; ++t) src_tok[T * k + t] = (int32_t)t;
    free(cursor);
}

/* -------------------------------------------------------------- expert FFN */

enum { ORC_MODE_F32 = 0, ORC_MODE_BF16 = 1, ORC_MODE_FP8 = 2 };

typedef struct {
    int32_t D, I, mode;
    const void *wg, *wu, *wd;          /* [G, I, D], [G, I, D], [G, D, I] */
    const float *sg, *su, *sd;         /* FP8 block scales, [G, I/128, D/128] etc. */
} experts_t;

/* Weight element (r, c) of group g's [rows, cols] matrix, as the value it
 * stands for. */
static inline double wval(const experts_t* ex, const void* base, const float* sc, int64_t g,
                          int64_t rows, int64_t cols, int64_t r, int64_t c) {
    int64_t i = g * rows * cols + r * cols + c;
    if (ex->mode == ORC_MODE_F32) return (double)((const float*)base)[i];
    if (ex->mode == ORC_MODE_BF16) return orc_bf16_to_f64(((const uint16_t*)base)[i]);
    double s = (double)sc[g * (rows / 128) * (cols / 128) + (r / 128) * (cols / 128) + c / 128];
    return orc_e4m3_to_f64(((const uint8_t*)base)[i]) * s;
}

/* SwiGLU expert g on one token: a = Wg x, u = Wu x, h = a * sigmoid(a) * u,
 * y = Wd h.  In FP8 mode the input row xin is already the dequantised E4M3
 * activation; h is rounded to fp32 and put through the 1 x 128 quantiser
 * before the down projection. */
static void expert_ffn(const experts_t* ex, int64_t g, const double* xin, double* h, float* hf,
                       double* hq, double* y) {
    const int64_t D = ex->D, I = ex->I;
    for (int64_t i = 0; i < I; ++i) {
        double a = 0.0, u = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            a += wval(ex, ex->wg, ex->sg, g, I, D, i, d) * xin[d];
            u += wval(ex, ex->wu, ex->su, g, I, D, i, d) * xin[d];
        }
        h[i] = a / (1.0 + exp(-a)) * u;
    }
    const double* hin = h;
    if (ex->mode == ORC_MODE_FP8) {
        for (int64_t i = 0; i < I; ++i) hf[i] = (float)h[i];
        quant_row_128(I, hf, hq);
        hin = hq;
    }
    for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i) acc += wval(ex, ex->wd, ex->sd, g, D, I, d, i) * hin[i];
        y[d] = acc;
    }
}

/* The layer for n tokens whose routing is given:
 *   out[t] = shared(x_t) + sum_j w[t,j] * expert_{idx[t,j]}(x_t).
 * Expert weights hold E+1 groups; group E is the shared expert.  x is fp32
 * (mode F32) or bf16 (modes BF16 and FP8; FP8 quantises it per token per
 * 128-column group first).  y_out (nullable) receives the k+1 expert outputs
 * of every token, [n, k+1, D], slot k being the shared expert's. */
ORC_EXPORT void orc_moe_tokens(int64_t n, int32_t D, int32_t E, int32_t I, int32_t k, int32_t mode,
                               const void* x, const int32_t* idx, const double* w, const void* wg,
                               const void* wu, const void* wd, const float* sg, const float* su,
                               const float* sd, double* out, double* y_out) {
    experts_t ex = {D, I, mode, wg, wu, wd, sg, su, sd};
    const int x_dt = (mode == ORC_MODE_F32) ? ORC_F32 : ORC_BF16;
#pragma omp parallel
    {
        double* xin = (double*)malloc(sizeof(double) * (size_t)D);
        float* xf = (float*)malloc(sizeof(float) * (size_t)D);
        double* h = (double*)malloc(sizeof(double) * (size_t)I);
        float* hf = (float*)malloc(sizeof(float) * (size_t)I);
        double* hq = (double*)malloc(sizeof(double) * (size_t)I);
        double* y = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n; ++t) {
            for (int64_t d = 0; d < D; ++d) xin[d] = load_elem(x_dt, x, t * D + d);
            if (mode == ORC_MODE_FP8) {
                for (int64_t d = 0; d < D; ++d) xf[d] = (float)xin[d];
                quant_row_128(D, xf, xin);
            }
            double* o = out + t * D;
            expert_ffn(&ex, E, xin, h, hf, hq, y);          /* shared expert, weight 1 */
            for (int64_t d = 0; d < D; ++d) o[d] = y[d];
            if (y_out) memcpy(y_out + (t * (k + 1) + k) * D, y, sizeof(double) * (size_t)D);
            for (int32_t j = 0; j < k; ++j) {
                expert_ffn(&ex, idx[t * k + j], xin, h, hf, hq, y);
                for (int64_t d = 0; d < D; ++d) o[d] += w[t * k + j] * y[d];
                if (y_out) memcpy(y_out + (t * (k + 1) + j) * D, y, sizeof(double) * (size_t)D);
            }
        }
        free(xin); free(xf); free(h); free(hf); free(hq); free(y);
    }
}

/* The whole layer from x: fp64 logits -> top-k -> experts -> combine.
 * idx_out [T,k] and w_out [T,k] receive the routing. */
ORC_EXPORT void orc_moe_layer(int64_t T, int32_t D, int32_t E, int32_t I, int32_t k, int32_t mode,
                              const void* x, const void* w_r, const float* bias, const void* wg,
                              const void* wu, const void* wd, const float* sg, const float* su,
                              const float* sd, double* out, int32_t* idx_out, double* w_out) {
    const int x_dt = (mode == ORC_MODE_F32) ? ORC_F32 : ORC_BF16;
    double* z = (double*)malloc(sizeof(double) * (size_t)(T * E));
    orc_logits(T, D, E, x_dt, x, x_dt, w_r, bias, z);
    orc_topk(T, E, k, z, idx_out, w_out);
    free(z);
    orc_moe_tokens(T, D, E, I, k, mode, x, idx_out, w_out, wg, wu, wd, sg, su, sd, out, NULL);
}

/* Blob of the pages' "Fusing Three Collectives Into Two": the [T,k] index
 * plane and the [T,k] weight plane stacked into one int32 buffer [2,T,k],
 * plane 1 holding the fp32 bit pattern of each weight. */
ORC_EXPORT void orc_pack_blob(int64_t T, int32_t k, const int32_t* idx, const float* w, int32_t* blob) {
    for (int64_t i = 0; i < T * k; ++i) {
        blob[i] = idx[i];
        memcpy(&blob[T * k + i], &w[i], 4);
    }
}

/* Compact one-word form of the same blob: bits 0..15 the expert index,
 * bits 16..31 the bf16 (round to nearest even) of the fp32 weight. */
ORC_EXPORT void orc_pack_words(int64_t T, int32_t k, const int32_t* idx, const float* w, int32_t* words) {
    for (int64_t i = 0; i < T * k; ++i) {
        uint32_t word = ((uint32_t)idx[i] & 0xFFFFu) | ((uint32_t)orc_f32_to_bf16(w[i]) << 16);
        memcpy(&words[i], &word, 4);
    }
}

/* Combine step on its own (unpermute): out[t] = y[T*k + t] + sum_j w[t,j] *
 * y[inv[t*k+j]], over rows y of the expert-contiguous layout, in double. */
ORC_EXPORT void orc_unpermute(int64_t T, int32_t D, int32_t k, const double* y, const double* w,
                              const int32_t* inv, double* out) {
    for (int64_t t = 0; t < T; ++t)
        for (int32_t d = 0; d < D; ++d) {
            double acc = y[(T * k + t) * D + d];
            for (int32_t j = 0; j < k; ++j) acc += w[t * k + j] * y[(int64_t)inv[t * k + j] * D + d];
            out[t * D + d] = acc;
        }
}

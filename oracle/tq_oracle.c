/*
 * tq_oracle.c -- CPU oracle (TEST INFRASTRUCTURE ONLY; see tq_oracle.h).
 *
 * Compiled with -O2 -ffp-contract=off so that every float operation below is
 * one IEEE binary32 (or binary64) operation with round-to-nearest-even, in
 * the order written.  No SIMD intrinsics, no fast-math.
 */
#include "tq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* binary16 codec, written from the IEEE 754 binary16 definition:            */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 means  */
/* subnormal (fraction * 2^-24), exponent 31 means Inf/NaN.                   */
/* ------------------------------------------------------------------------ */

double tqo_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f | 0x400), e - 25); /* (1024 + f) * 2^(e - 15 - 10) */
    }
    return sign ? -v : v;
}

uint16_t tqo_f32_to_f16(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t e32 = (u >> 23) & 0xffu;
    uint32_t f32 = u & 0x7fffffu;
    if (e32 == 0xffu) { /* Inf or NaN (NaN keeps a quiet payload bit) */
        return (uint16_t)(sign | 0x7c00u | (f32 ? 0x200u : 0u));
    }
    if (e32 == 0) { /* binary32 zero/subnormal: magnitude < 2^-126 -> 0 */
        return sign;
    }
    int e = (int)e32 - 127;            /* value = 1.f * 2^e */
    uint32_t sig = f32 | 0x800000u;     /* 24-bit significand, value = sig * 2^(e-23) */
    if (e >= -14) {
        if (e > 15) return (uint16_t)(sign | 0x7c00u); /* overflow -> Inf */
        /* normal binary16: keep 11 significant bits, drop 13, round RNE */
        uint32_t keep = sig >> 13;
        uint32_t rest = sig & 0x1fffu;
        uint32_t h = ((uint32_t)(e + 15) << 10) | (keep & 0x3ffu);
        if (rest > 0x1000u || (rest == 0x1000u && (keep & 1u))) h += 1u; /* may carry into exponent */
        return (uint16_t)(sign | h);     /* carry past 0x7bff gives 0x7c00 = Inf, as RNE demands */
    }
    /* subnormal binary16: units of 2^-24, count = sig * 2^(e - 23 + 24) */
    int shift = -(e + 1);               /* >= 14 here */
    if (shift > 24) return sign;        /* below 2^-25: rounds to zero */
    uint32_t keep = sig >> shift;
    uint32_t rest = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rest > half || (rest == half && (keep & 1u))) keep += 1u; /* may reach 0x400 = min normal */
    return (uint16_t)(sign | keep);
}

void tqo_f32_to_f16_array(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = tqo_f32_to_f16(x[i]);
}

void tqo_f16_to_f64_array(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = tqo_f16_to_f64(h[i]);
}

/* ------------------------------------------------------------------------ */
/* Affine int4 quantisation of one group ([G4] Background: per-group scale +  */
/* bias; [TQ] group 64).  Steps in the order fixed by the header.             */
/* ------------------------------------------------------------------------ */

/* levels = 2^bits - 1 codes above zero: 15 for int4 ([G4] Background), 255
 * for int8 ([TQ] driver flag --kv-bits {4,8}); the same affine rule. */
void tqo_quantize_group_b(const uint16_t* x, int n, int bits, uint8_t* codes,
                          uint16_t* scale, uint16_t* bias) {
    const float levels = (float)((1 << bits) - 1);
    float mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < n; ++i) {
        float xi = (float)tqo_f16_to_f64(x[i]); /* exact: every fp16 is a float */
        if (xi < mn) mn = xi;
        if (xi > mx) mx = xi;
    }
    if (mn == 0.0f) mn = 0.0f;               /* a zero minimum is stored as +0 */
    volatile float range = mx - mn;          /* one binary32 subtraction */
    volatile float s32 = range / levels;     /* one binary32 division */
    uint16_t sh = tqo_f32_to_f16(s32);
    uint16_t bh = tqo_f32_to_f16(mn);        /* exact: mn is an fp16 value */
    float s = (float)tqo_f16_to_f64(sh);
    float b = (float)tqo_f16_to_f64(bh);
    *scale = sh;
    *bias = bh;
    for (int i = 0; i < n; ++i) {
        if (s == 0.0f) {
            codes[i] = 0;
            continue;
        }
        float xi = (float)tqo_f16_to_f64(x[i]);
        volatile float d = xi - b;           /* binary32 subtraction */
        volatile float t = d / s;            /* binary32 division */
        float r = rintf(t);                  /* default rounding mode: nearest-even */
        if (r < 0.0f) r = 0.0f;
        if (r > levels) r = levels;
        codes[i] = (uint8_t)r;
    }
}

void tqo_quantize_group(const uint16_t* x, int n, uint8_t* codes,
                        uint16_t* scale, uint16_t* bias) {
    tqo_quantize_group_b(x, n, 4, codes, scale, bias);
}

/* int4: two codes per byte (element 2i in the low nibble of byte i); int8:
 * one code per byte. */
void tqo_quantize_rows_b(const uint16_t* x, int64_t rows, int D, int group, int bits,
                         uint8_t* codes_packed, uint16_t* scale, uint16_t* bias) {
    int ng = D / group;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        uint8_t codes[1024];
        for (int g = 0; g < ng; ++g) {
            tqo_quantize_group_b(x + r * D + (int64_t)g * group, group, bits, codes + g * group,
                                 scale + r * ng + g, bias + r * ng + g);
        }
        if (bits == 8) {
            for (int i = 0; i < D; ++i) codes_packed[r * D + i] = codes[i];
            continue;
        }
        for (int i = 0; i < D / 2; ++i) {
            /* [G4] masks 0xF then 0xF0: the earlier element sits in the low nibble */
            codes_packed[r * (D / 2) + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
        }
    }
}

void tqo_quantize_rows(const uint16_t* x, int64_t rows, int D, int group,
                       uint8_t* codes_packed, uint16_t* scale, uint16_t* bias) {
    tqo_quantize_rows_b(x, rows, D, group, 4, codes_packed, scale, bias);
}

static double dequant_one_b(const uint8_t* row_codes, const uint16_t* row_scale,
                            const uint16_t* row_bias, int d, int group, int bits) {
    int code;
    if (bits == 8) {
        code = row_codes[d];
    } else {
        uint8_t byte = row_codes[d / 2];
        code = (d & 1) ? (byte >> 4) : (byte & 0xf);
    }
    int g = d / group;
    return tqo_f16_to_f64(row_scale[g]) * (double)code + tqo_f16_to_f64(row_bias[g]);
}

static double dequant_one(const uint8_t* row_codes, const uint16_t* row_scale,
                          const uint16_t* row_bias, int d, int group) {
    return dequant_one_b(row_codes, row_scale, row_bias, d, group, 4);
}

void tqo_dequantize_rows_b(const uint8_t* codes_packed, const uint16_t* scale,
                           const uint16_t* bias, int64_t rows, int D, int group, int bits,
                           double* out) {
    int ng = D / group;
    int64_t row_bytes = (int64_t)D * bits / 8;
    for (int64_t r = 0; r < rows; ++r)
        for (int d = 0; d < D; ++d)
            out[r * D + d] = dequant_one_b(codes_packed + r * row_bytes, scale + r * ng,
                                           bias + r * ng, d, group, bits);
}

void tqo_dequantize_rows(const uint8_t* codes_packed, const uint16_t* scale,
                         const uint16_t* bias, int64_t rows, int D, int group,
                         double* out) {
    tqo_dequantize_rows_b(codes_packed, scale, bias, rows, D, group, 4, out);
}

/* fp16 dequantisation: the float K/V a dequantize-then-SDPA baseline builds
 * before attention ([G4] What I Built Instead: the MLX path expands the int4
 * cache to float K/V and runs ordinary SDPA).  Reading: one fp32 rounding of
 * scale * code + bias (the product is exact in fp32: 11 x 4 significant bits),
 * then RNE to binary16. */
void tqo_dequantize_rows_f16_b(const uint8_t* codes_packed, const uint16_t* scale,
                               const uint16_t* bias, int64_t rows, int D, int group, int bits,
                               uint16_t* out) {
    int ng = D / group;
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* rc = codes_packed + r * ((int64_t)D * bits / 8);
        for (int d = 0; d < D; ++d) {
            int code;
            if (bits == 8) {
                code = rc[d];
            } else {
                uint8_t byte = rc[d / 2];
                code = (d & 1) ? (byte >> 4) : (byte & 0xf);
            }
            int g = d / group;
            float sc = (float)tqo_f16_to_f64(scale[r * ng + g]);
            float bi = (float)tqo_f16_to_f64(bias[r * ng + g]);
            out[r * D + d] = tqo_f32_to_f16(fmaf(sc, (float)code, bi));
        }
    }
}

void tqo_dequantize_rows_f16(const uint8_t* codes_packed, const uint16_t* scale,
                             const uint16_t* bias, int64_t rows, int D, int group,
                             uint16_t* out) {
    tqo_dequantize_rows_f16_b(codes_packed, scale, bias, rows, D, group, 4, out);
}

/* ------------------------------------------------------------------------ */
/* Hadamard rotation ([TQ] "Running and Evaluating TurboQuant optimized       */
/* Gemma 4": the key breakthrough paragraph and the worked example -- a       */
/* normalised Sylvester Hadamard matrix H / sqrt(n) spreads an outlier over  */
/* all coordinates before quantisation and, being its own inverse, brings    */
/* the vector back).  y = (1/sqrt(n)) * H_n x with H_1 = [1], H_2m =          */
/* [[H_m, H_m], [H_m, -H_m]], evaluated as the fast transform: for h = 1, 2,  */
/* 4, ..., n/2, every pair (i, i + h) with bit h of i clear becomes           */
/* (x_i + x_{i+h}, x_i - x_{i+h}); then every element is multiplied by        */
/* 1/sqrt(n).  Readings: the fp32 variant performs exactly these operations  */
/* in fp32 (the stage order fixes the rounding), with 1/sqrt(n) taken as the */
/* fp32 value nearest to the fp64 1/sqrt(n); the rows variant converts fp16  */
/* input to fp32 and rounds the result to fp16 (RNE).                        */
/* ------------------------------------------------------------------------ */

static int is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

void tqo_hadamard_f64(double* x, int n) {
    if (!is_pow2(n)) return;
    for (int h = 1; h < n; h <<= 1)
        for (int i = 0; i < n; ++i)
            if ((i & h) == 0) {
                double u = x[i], v = x[i + h];
                x[i] = u + v;
                x[i + h] = u - v;
            }
    double c = 1.0 / sqrt((double)n);
    for (int i = 0; i < n; ++i) x[i] *= c;
}

void tqo_hadamard_f32(float* x, int n) {
    if (!is_pow2(n)) return;
    for (int h = 1; h < n; h <<= 1)
        for (int i = 0; i < n; ++i)
            if ((i & h) == 0) {
                float u = x[i], v = x[i + h];
                x[i] = u + v;
                x[i + h] = u - v;
            }
    float c = (float)(1.0 / sqrt((double)n));
    for (int i = 0; i < n; ++i) x[i] *= c;
}

void tqo_rotate_rows_f16(const uint16_t* x, int64_t rows, int n, uint16_t* out) {
    float buf[1024];
    if (!is_pow2(n) || n > 1024) return;
    for (int64_t r = 0; r < rows; ++r) {
        for (int i = 0; i < n; ++i) buf[i] = (float)tqo_f16_to_f64(x[r * n + i]);
        tqo_hadamard_f32(buf, n);
        for (int i = 0; i < n; ++i) out[r * n + i] = tqo_f32_to_f16(buf[i]);
    }
}

/* ------------------------------------------------------------------------ */
/* Decode attention ([L70] kernel paragraph: scores from the int4 data,       */
/* softmax, weighted sum of values; GQA with Hq/Hkv query heads per KV head). */
/* The oracle simply dequantises and runs ordinary attention in fp64.         */
/* ------------------------------------------------------------------------ */

typedef struct {
    int B, Hq, Hkv, D, group;
    int64_t cap;
    const uint8_t *kc, *vc;
    const uint16_t *ks, *kb, *vs, *vb;
    int bits; /* 4: two codes per byte; 8: one */
} cache_view;

static void row_ptrs(const cache_view* c, int b, int kvh, int64_t t,
                     const uint8_t** codes, const uint16_t** s, const uint16_t** bi, int is_v) {
    int ng = c->D / c->group;
    int64_t row = ((int64_t)b * c->Hkv + kvh) * c->cap + t;
    *codes = (is_v ? c->vc : c->kc) + row * ((int64_t)c->D * c->bits / 8);
    *s = (is_v ? c->vs : c->ks) + row * ng;
    *bi = (is_v ? c->vb : c->kb) + row * ng;
}

/* score s_t = attn_scale * sum_d q[d] * khat[t][d] */
static double score(const cache_view* c, const double* qd, int b, int kvh, int64_t t,
                    double attn_scale) {
    const uint8_t* codes;
    const uint16_t *s, *bi;
    row_ptrs(c, b, kvh, t, &codes, &s, &bi, 0);
    double acc = 0.0;
    for (int d = 0; d < c->D; ++d) acc += qd[d] * dequant_one_b(codes, s, bi, d, c->group, c->bits);
    return attn_scale * acc;
}

static void add_weighted_v(const cache_view* c, int b, int kvh, int64_t t, double w,
                           double* acc) {
    const uint8_t* codes;
    const uint16_t *s, *bi;
    row_ptrs(c, b, kvh, t, &codes, &s, &bi, 1);
    for (int d = 0; d < c->D; ++d) acc[d] += w * dequant_one_b(codes, s, bi, d, c->group, c->bits);
}

static void attend_one(const cache_view* c, const uint16_t* q, int b, int h, int64_t len,
                       double attn_scale, double* out_row) {
    int G = c->Hq / c->Hkv;
    int kvh = h / G;
    double* qd = (double*)malloc(sizeof(double) * c->D);
    for (int d = 0; d < c->D; ++d)
        qd[d] = tqo_f16_to_f64(q[((int64_t)b * c->Hq + h) * c->D + d]);
    for (int d = 0; d < c->D; ++d) out_row[d] = 0.0;
    if (len <= 0) {
        free(qd);
        return;
    }
    double* sc = (double*)malloc(sizeof(double) * (size_t)len);
    double m = -INFINITY;
    for (int64_t t = 0; t < len; ++t) {
        sc[t] = score(c, qd, b, kvh, t, attn_scale);
        if (sc[t] > m) m = sc[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < len; ++t) {
        double p = exp(sc[t] - m);
        l += p;
        add_weighted_v(c, b, kvh, t, p, out_row);
    }
    for (int d = 0; d < c->D; ++d) out_row[d] /= l;
    free(sc);
    free(qd);
}

void tqo_attention_b(const uint16_t* q, int B, int Hq, int Hkv, int D, int group,
                     int64_t cap, const uint8_t* kc, const uint16_t* ks,
                     const uint16_t* kb, const uint8_t* vc, const uint16_t* vs,
                     const uint16_t* vb, const int32_t* lens, double attn_scale,
                     const int32_t* pairs, int64_t n_pairs, int bits, double* out) {
    cache_view c = {B, Hq, Hkv, D, group, cap, kc, vc, ks, kb, vs, vb, bits};
    int64_t n = pairs ? n_pairs : (int64_t)B * Hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < n; ++i) {
        int b = pairs ? pairs[2 * i] : (int)(i / Hq);
        int h = pairs ? pairs[2 * i + 1] : (int)(i % Hq);
        attend_one(&c, q, b, h, lens[b], attn_scale, out + ((int64_t)b * Hq + h) * D);
    }
}

void tqo_attention(const uint16_t* q, int B, int Hq, int Hkv, int D, int group,
                   int64_t cap, const uint8_t* kc, const uint16_t* ks,
                   const uint16_t* kb, const uint8_t* vc, const uint16_t* vs,
                   const uint16_t* vb, const int32_t* lens, double attn_scale,
                   const int32_t* pairs, int64_t n_pairs, double* out) {
    tqo_attention_b(q, B, Hq, Hkv, D, group, cap, kc, ks, kb, vc, vs, vb, lens, attn_scale, pairs,
                    n_pairs, 4, out);
}

/* ------------------------------------------------------------------------ */
/* Split-K ([L70] split-K paragraph): phase 1 emits, per 512-token chunk, the */
/* partial softmax state (max m, sum l, unnormalised weighted sum acc);       */
/* phase 2 reduces the partials with a log-sum-exp merge.                     */
/* ------------------------------------------------------------------------ */

void tqo_attention_partials_b(const uint16_t* q, int B, int Hq, int Hkv, int D,
                              int group, int64_t cap, const uint8_t* kc,
                              const uint16_t* ks, const uint16_t* kb,
                              const uint8_t* vc, const uint16_t* vs,
                              const uint16_t* vb, const int32_t* lens,
                              double attn_scale, int chunk, int n_chunks, int bits,
                              double* part_m, double* part_l, double* part_acc) {
    cache_view c = {B, Hq, Hkv, D, group, cap, kc, vc, ks, kb, vs, vb, bits};
    int G = Hq / Hkv;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < (int64_t)B * Hq; ++i) {
        int b = (int)(i / Hq), h = (int)(i % Hq), kvh = h / G;
        double* qd = (double*)malloc(sizeof(double) * D);
        for (int d = 0; d < D; ++d) qd[d] = tqo_f16_to_f64(q[i * D + d]);
        for (int ci = 0; ci < n_chunks; ++ci) {
            int64_t t0 = (int64_t)ci * chunk, t1 = t0 + chunk;
            if (t1 > lens[b]) t1 = lens[b];
            double* acc = part_acc + (i * n_chunks + ci) * D;
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            double m = -INFINITY, l = 0.0;
            for (int64_t t = t0; t < t1; ++t) {
                double s = score(&c, qd, b, kvh, t, attn_scale);
                if (s > m) m = s;
            }
            for (int64_t t = t0; t < t1; ++t) {
                double p = exp(score(&c, qd, b, kvh, t, attn_scale) - m);
                l += p;
                add_weighted_v(&c, b, kvh, t, p, acc);
            }
            part_m[i * n_chunks + ci] = m;
            part_l[i * n_chunks + ci] = l;
        }
        free(qd);
    }
}

void tqo_attention_partials(const uint16_t* q, int B, int Hq, int Hkv, int D,
                            int group, int64_t cap, const uint8_t* kc,
                            const uint16_t* ks, const uint16_t* kb,
                            const uint8_t* vc, const uint16_t* vs,
                            const uint16_t* vb, const int32_t* lens,
                            double attn_scale, int chunk, int n_chunks,
                            double* part_m, double* part_l, double* part_acc) {
    tqo_attention_partials_b(q, B, Hq, Hkv, D, group, cap, kc, ks, kb, vc, vs, vb, lens, attn_scale, chunk,
                             n_chunks, 4, part_m, part_l, part_acc);
}

void tqo_merge_partials(const double* part_m, const double* part_l,
                        const double* part_acc, int B, int Hq, int D,
                        int n_chunks, double* out) {
    for (int64_t i = 0; i < (int64_t)B * Hq; ++i) {
        double M = -INFINITY;
        for (int ci = 0; ci < n_chunks; ++ci)
            if (part_l[i * n_chunks + ci] > 0.0 && part_m[i * n_chunks + ci] > M)
                M = part_m[i * n_chunks + ci];
        double L = 0.0;
        for (int d = 0; d < D; ++d) out[i * D + d] = 0.0;
        if (M == -INFINITY) continue; /* every chunk empty: zero row */
        for (int ci = 0; ci < n_chunks; ++ci) {
            double l = part_l[i * n_chunks + ci];
            if (!(l > 0.0)) continue;
            double w = exp(part_m[i * n_chunks + ci] - M);
            L += w * l;
            for (int d = 0; d < D; ++d) out[i * D + d] += w * part_acc[(i * n_chunks + ci) * D + d];
        }
        for (int d = 0; d < D; ++d) out[i * D + d] /= L;
    }
}

int tqo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * tq_oracle.h -- CPU oracle for int4 KV-cache quantize-on-store and fused
 * decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously-correct C with fp64
 * accumulation.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call it; the product path never
 * does.  It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (the pages this restates):
 *   [G4]  "Fused int4 Attention for Gemma 4 31B on Apple Silicon",
 *         sections "Background" and "What I Built Instead"
 *         (per-group scale + bias int4; sdpa_int4(Q, K_int4, V_int4);
 *          uint16 nibble masks 0xF, 0xF0, 0xF00, 0xF000 -> low nibble first).
 *   [L70] "turboquant-llama3.170B" README: kernel paragraph (online softmax,
 *         no S x S matrix), kernel latency table (64 q / 8 kv heads),
 *         split-K paragraph (512-token chunks, partial softmax, reduce),
 *         decode-step listing (RoPE -> quantize K,V to int4 -> fused sdpa_int4).
 *   [TQ]  "Running and Evaluating TurboQuant optimized Gemma 4": --kv-bits 4,
 *         --kv-group-size 64 defaults.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - affine int4: x ~ scale * q + bias, q in [0, 15], bias = group min,
 *     scale = (max - min) / 15, group = 64 consecutive head_dim elements,
 *     scale and bias stored as fp16;
 *   - op order fixed for bit-exactness: min/max in fp32 (exact), r = fp32(max -
 *     min), s32 = fp32(r / 15), scale = fp16_rne(s32), bias = fp16(min) (exact),
 *     code = clamp(rint_rne(fp32(fp32(x - bias) / float(scale))), 0, 15), and
 *     code = 0 for every element when float(scale) == 0; a group whose minimum
 *     is zero stores bias +0 whatever the sign of its zeros (so that the bias
 *     bits do not depend on the order in which the minimum is searched);
 *   - codes packed two per byte, element 2i in the low nibble of byte i;
 *   - dequantised value = (double)scale * code + (double)bias;
 *   - GQA: query head h reads KV head h / (Hq / Hkv);
 *   - no mask, no softcap: decode attends to all of [0, len);
 *   - len == 0 gives an all-zero output row.
 *
 * Parity status: every function below is pinned by tests that do not reuse
 * its arithmetic (see tests/test_oracle_pins.py).
 */
#ifndef TQ_ORACLE_H
#define TQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE binary16 <-> binary32/binary64 codec (RNE for the narrowing). */
uint16_t tqo_f32_to_f16(float x);
double tqo_f16_to_f64(uint16_t h);
void tqo_f32_to_f16_array(const float* x, int64_t n, uint16_t* out);
void tqo_f16_to_f64_array(const uint16_t* h, int64_t n, double* out);

/* Quantize one group of n fp16 values: codes[n] unpacked (0..15). */
void tqo_quantize_group(const uint16_t* x, int n, uint8_t* codes,
                        uint16_t* scale, uint16_t* bias);

/* Quantize `rows` rows of D fp16 values (groups of `group` along the row).
 * codes_packed: [rows][D/2] (element 2i -> low nibble of byte i)
 * scale, bias:  [rows][D/group] fp16 bits. */
void tqo_quantize_rows(const uint16_t* x, int64_t rows, int D, int group,
                       uint8_t* codes_packed, uint16_t* scale, uint16_t* bias);

/* Dequantize rows back to fp64: out[rows][D]. */
void tqo_dequantize_rows(const uint8_t* codes_packed, const uint16_t* scale,
                         const uint16_t* bias, int64_t rows, int D, int group,
                         double* out);

/* Dequantize rows to fp16 bits: out[rows][D] = fp16_rne(fp32(scale * code + bias)),
 * the float cache of a dequantize-then-attend baseline. */
void tqo_dequantize_rows_f16(const uint8_t* codes_packed, const uint16_t* scale,
                             const uint16_t* bias, int64_t rows, int D, int group,
                             uint16_t* out);

/* The same with a code width: bits = 4 (levels 15, two codes per byte) or 8
 * (levels 255, one code per byte); the functions above are bits = 4. */
void tqo_quantize_group_b(const uint16_t* x, int n, int bits, uint8_t* codes,
                          uint16_t* scale, uint16_t* bias);
void tqo_quantize_rows_b(const uint16_t* x, int64_t rows, int D, int group, int bits,
                         uint8_t* codes_packed, uint16_t* scale, uint16_t* bias);
void tqo_dequantize_rows_f16_b(const uint8_t* codes_packed, const uint16_t* scale,
                               const uint16_t* bias, int64_t rows, int D, int group, int bits,
                               uint16_t* out);
void tqo_dequantize_rows_b(const uint8_t* codes_packed, const uint16_t* scale,
                           const uint16_t* bias, int64_t rows, int D, int group, int bits,
                           double* out);
void tqo_attention_b(const uint16_t* q, int B, int Hq, int Hkv, int D, int group,
                     int64_t cap, const uint8_t* kc, const uint16_t* ks,
                     const uint16_t* kb, const uint8_t* vc, const uint16_t* vs,
                     const uint16_t* vb, const int32_t* lens, double attn_scale,
                     const int32_t* pairs, int64_t n_pairs, int bits, double* out);

/* Normalised Sylvester Hadamard transform in place, n a power of two:
 * x <- (1/sqrt(n)) H_n x by the fast transform (stages h = 1, 2, ..., n/2).
 * The f64 form is the reference; the f32 form performs the same operations in
 * fp32 (the rotation applied to K and Q before quantisation / attention). */
void tqo_hadamard_f64(double* x, int n);
void tqo_hadamard_f32(float* x, int n);
/* Rotate fp16 rows: out = fp16_rne(fp32 transform of the fp16 row), n <= 1024. */
void tqo_rotate_rows_f16(const uint16_t* x, int64_t rows, int n, uint16_t* out);

/* Single-token decode attention over a quantised cache.
 * q:    [B][Hq][D] fp16 bits
 * kc,vc:[B][Hkv][cap][D/2] packed codes; ks,kb,vs,vb: [B][Hkv][cap][D/group]
 * lens: [B] tokens attended per sequence (0 <= lens[b] <= cap)
 * pairs:optional list of n_pairs (b, h) pairs to compute (NULL = all B*Hq);
 *       rows of `out` not in the list are left untouched.
 * out:  [B][Hq][D] fp64.
 * Two-pass softmax in fp64: m = max_t s_t, p_t = exp(s_t - m),
 * out = sum_t p_t v_t / sum_t p_t. */
void tqo_attention(const uint16_t* q, int B, int Hq, int Hkv, int D, int group,
                   int64_t cap, const uint8_t* kc, const uint16_t* ks,
                   const uint16_t* kb, const uint8_t* vc, const uint16_t* vs,
                   const uint16_t* vb, const int32_t* lens, double attn_scale,
                   const int32_t* pairs, int64_t n_pairs, double* out);

/* Split-K phase 1 (per chunk of `chunk` tokens starting at token 0):
 * part_m[B][Hq][nc]  = max score in the chunk (-inf if the chunk is empty)
 * part_l[B][Hq][nc]  = sum exp(s - m)          (0 if empty)
 * part_acc[B][Hq][nc][D] = sum exp(s - m) v_t   (0 if empty)
 * with nc = n_chunks (callers pass ceil(max_len / chunk)). */
void tqo_attention_partials(const uint16_t* q, int B, int Hq, int Hkv, int D,
                            int group, int64_t cap, const uint8_t* kc,
                            const uint16_t* ks, const uint16_t* kb,
                            const uint8_t* vc, const uint16_t* vs,
                            const uint16_t* vb, const int32_t* lens,
                            double attn_scale, int chunk, int n_chunks,
                            double* part_m, double* part_l, double* part_acc);
/* The same for a cache of `bits`-bit codes (4 or 8: "Running and Evaluating
 * TurboQuant optimized Gemma 4", driver flags --kv-bits {4,8}). */
void tqo_attention_partials_b(const uint16_t* q, int B, int Hq, int Hkv, int D,
                              int group, int64_t cap, const uint8_t* kc,
                              const uint16_t* ks, const uint16_t* kb,
                              const uint8_t* vc, const uint16_t* vs,
                              const uint16_t* vb, const int32_t* lens,
                              double attn_scale, int chunk, int n_chunks, int bits,
                              double* part_m, double* part_l, double* part_acc);

/* Split-K phase 2: log-sum-exp merge of n_chunks partials per (b, h).
 * out[B][Hq][D] = sum_c e^{m_c - M} acc_c / sum_c e^{m_c - M} l_c,
 * M = max_c m_c; chunks with l == 0 are skipped; all-empty rows give 0. */
void tqo_merge_partials(const double* part_m, const double* part_l,
                        const double* part_acc, int B, int Hq, int D,
                        int n_chunks, double* out);

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int tqo_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ_ORACLE_H */

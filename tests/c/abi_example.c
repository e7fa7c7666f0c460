/*
 * abi_example.c -- the C ABI used from plain C (no Python, no PyTorch): quantize
 * a cache, decode, run one fused step, and check everything against the CPU
 * oracle.  Test infrastructure (it links the oracle); tests/test_c_abi.py
 * compiles and runs it.
 *
 * Exit status 0 and a line "OK ..." when the codes, scales and biases equal the
 * oracle's bit for bit and the outputs are within 2e-3 max-abs and 1e-3
 * relative L2 of the oracle's fp64 attention; 1 otherwise (with the reason).
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "tq.h"
#include "tq_oracle.h"

#define CHECK_CUDA(x)                                                         \
    do {                                                                      \
        cudaError_t e_ = (x);                                                 \
        if (e_ != cudaSuccess) {                                              \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));          \
            return 1;                                                         \
        }                                                                     \
    } while (0)
#define CHECK_TQ(x)                                                           \
    do {                                                                      \
        tq_status s_ = (x);                                                   \
        if (s_ != TQ_OK) {                                                    \
            fprintf(stderr, "%s: %s\n", #x, tq_status_string(s_));            \
            return 1;                                                         \
        }                                                                     \
    } while (0)

enum { B = 2, HQ = 16, HKV = 2, D = 128, G64 = 64, CAP = 1024 };

/* Seeded standard-normal-ish values (sum of four uniforms, centred and
 * scaled to unit variance) from a 64-bit LCG. */
static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static double uniform01(void) {
    rng_state = rng_state * 6364136223846793005ull + 1442695040888963407ull;
    return (double)(rng_state >> 11) * (1.0 / 9007199254740992.0);
}
static float draw(void) {
    double s = uniform01() + uniform01() + uniform01() + uniform01() - 2.0;
    return (float)(s * sqrt(3.0));
}

static void fill_f16(uint16_t* x, size_t n) {
    for (size_t i = 0; i < n; ++i) x[i] = tqo_f32_to_f16(draw());
}

static int compare_out(const char* what, const uint16_t* got, const double* ref, size_t n) {
    double mx = 0.0, num = 0.0, den = 0.0;
    for (size_t i = 0; i < n; ++i) {
        const double g = tqo_f16_to_f64(got[i]), e = g - ref[i];
        if (!isfinite(g)) {
            fprintf(stderr, "%s: non-finite output at %zu\n", what, i);
            return 1;
        }
        if (fabs(e) > mx) mx = fabs(e);
        num += e * e;
        den += ref[i] * ref[i];
    }
    const double rel = den > 0.0 ? sqrt(num / den) : sqrt(num);
    printf("%s: max abs %.3e, rel L2 %.3e\n", what, mx, rel);
    if (mx > 2e-3 || rel > 1e-3) {
        fprintf(stderr, "%s: outside the tolerance\n", what);
        return 1;
    }
    return 0;
}

int main(void) {
    const int32_t lens_h[B] = {1000, 377};
    const int32_t max_len = 1000;
    const float attn = 1.0f / sqrtf((float)D);
    const size_t rows = (size_t)B * HKV * CAP, qn = (size_t)B * HQ * D;
    const int ng = D / G64;

    if (tq_abi_version() != TQ_ABI_VERSION) {
        fprintf(stderr, "ABI version mismatch\n");
        return 1;
    }
    uint16_t* k = malloc(rows * D * 2);
    uint16_t* v = malloc(rows * D * 2);
    uint16_t* q = malloc(qn * 2);
    uint16_t* out = malloc(qn * 2);
    uint16_t* kn = malloc((size_t)B * HKV * D * 2);
    uint16_t* vn = malloc((size_t)B * HKV * D * 2);
    uint8_t* kc = malloc(rows * D / 2);
    uint8_t* vc = malloc(rows * D / 2);
    uint16_t *ks = malloc(rows * ng * 2), *kb = malloc(rows * ng * 2);
    uint16_t *vs = malloc(rows * ng * 2), *vb = malloc(rows * ng * 2);
    uint8_t* gpu_codes = malloc(rows * D / 2);
    uint16_t* gpu_sb = malloc(rows * ng * 2);
    double* ref = malloc(qn * sizeof(double));
    if (!k || !v || !q || !out || !kn || !vn || !kc || !vc || !ks || !kb || !vs || !vb || !gpu_codes || !gpu_sb ||
        !ref)
        return 1;
    fill_f16(k, rows * D);
    fill_f16(v, rows * D);
    fill_f16(q, qn);
    fill_f16(kn, (size_t)B * HKV * D);
    fill_f16(vn, (size_t)B * HKV * D);

    /* cache: one device allocation carved into the six arrays */
    const size_t cache_bytes = tq_kv_cache_bytes(B, HKV, D, G64, CAP);
    void* base = NULL;
    CHECK_CUDA(cudaMalloc(&base, cache_bytes));
    tq_kv_cache cache;
    CHECK_TQ(tq_kv_cache_carve(&cache, base, B, HKV, D, G64, CAP));

    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));
    uint16_t *d_k, *d_v, *d_q, *d_out, *d_kn, *d_vn;
    int32_t *d_wp, *d_lens;
    CHECK_CUDA(cudaMalloc((void**)&d_k, rows * D * 2));
    CHECK_CUDA(cudaMalloc((void**)&d_v, rows * D * 2));
    CHECK_CUDA(cudaMalloc((void**)&d_q, qn * 2));
    CHECK_CUDA(cudaMalloc((void**)&d_out, qn * 2));
    CHECK_CUDA(cudaMalloc((void**)&d_kn, (size_t)B * HKV * D * 2));
    CHECK_CUDA(cudaMalloc((void**)&d_vn, (size_t)B * HKV * D * 2));
    CHECK_CUDA(cudaMalloc((void**)&d_wp, B * sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc((void**)&d_lens, B * sizeof(int32_t)));
    CHECK_CUDA(cudaMemcpy(d_k, k, rows * D * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_v, v, rows * D * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_q, q, qn * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_kn, kn, (size_t)B * HKV * D * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_vn, vn, (size_t)B * HKV * D * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_lens, lens_h, sizeof lens_h, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemset(d_wp, 0, B * sizeof(int32_t)));

    /* quantize all CAP rows of every (sequence, kv head) */
    CHECK_TQ(tq_quantize_kv_append(&cache, d_k, d_v, CAP, d_wp, NULL, stream));
    /* decode */
    const size_t ws_bytes = tq_sdpa_workspace_bytes(B, HQ, HKV, D, max_len, TQ_DEFAULT_CHUNK);
    void* ws = NULL;
    CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
    CHECK_TQ(tq_sdpa_int4_decode(&cache, d_q, HQ, d_lens, max_len, attn, TQ_DEFAULT_CHUNK, ws, ws_bytes, d_out, NULL,
                                 stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));
    CHECK_CUDA(cudaMemcpy(out, d_out, qn * 2, cudaMemcpyDeviceToHost));

    /* the oracle's cache, and the GPU's compared bit for bit */
    tqo_quantize_rows(k, (int64_t)rows, D, G64, kc, ks, kb);
    tqo_quantize_rows(v, (int64_t)rows, D, G64, vc, vs, vb);
    const struct {
        const void* dev;
        const void* want;
        size_t bytes;
        const char* name;
    } arrays[6] = {{cache.k_codes, kc, rows * D / 2, "k codes"}, {cache.k_scale, ks, rows * ng * 2, "k scale"},
                   {cache.k_bias, kb, rows * ng * 2, "k bias"},  {cache.v_codes, vc, rows * D / 2, "v codes"},
                   {cache.v_scale, vs, rows * ng * 2, "v scale"}, {cache.v_bias, vb, rows * ng * 2, "v bias"}};
    for (int i = 0; i < 6; ++i) {
        void* host = i % 3 == 0 ? (void*)gpu_codes : (void*)gpu_sb;
        CHECK_CUDA(cudaMemcpy(host, arrays[i].dev, arrays[i].bytes, cudaMemcpyDeviceToHost));
        if (memcmp(host, arrays[i].want, arrays[i].bytes) != 0) {
            fprintf(stderr, "%s differ from the oracle\n", arrays[i].name);
            return 1;
        }
    }
    tqo_attention(q, B, HQ, HKV, D, G64, CAP, kc, ks, kb, vc, vs, vb, lens_h, attn, NULL, 0, ref);
    if (compare_out("decode", out, ref, qn)) return 1;

    /* one fused step: append one token at row lens[b], attend over lens[b] + 1 */
    int32_t wp_h[B], lens1[B];
    for (int b = 0; b < B; ++b) {
        wp_h[b] = lens_h[b];
        lens1[b] = lens_h[b] + 1;
    }
    CHECK_CUDA(cudaMemcpy(d_wp, wp_h, sizeof wp_h, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_lens, lens1, sizeof lens1, cudaMemcpyHostToDevice));
    CHECK_TQ(tq_decode_step(&cache, d_kn, d_vn, 1, d_wp, d_q, HQ, d_lens, max_len + 1, attn, TQ_DEFAULT_CHUNK, ws,
                            ws_bytes, d_out, NULL, stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));
    CHECK_CUDA(cudaMemcpy(out, d_out, qn * 2, cudaMemcpyDeviceToHost));
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < HKV; ++h) {
            const size_t row = ((size_t)b * HKV + h) * CAP + (size_t)wp_h[b];
            memcpy(k + row * D, kn + ((size_t)b * HKV + h) * D, D * 2);
            memcpy(v + row * D, vn + ((size_t)b * HKV + h) * D, D * 2);
        }
    tqo_quantize_rows(k, (int64_t)rows, D, G64, kc, ks, kb);
    tqo_quantize_rows(v, (int64_t)rows, D, G64, vc, vs, vb);
    CHECK_CUDA(cudaMemcpy(gpu_codes, cache.k_codes, rows * D / 2, cudaMemcpyDeviceToHost));
    if (memcmp(gpu_codes, kc, rows * D / 2) != 0) {
        fprintf(stderr, "k codes after the step differ from the oracle\n");
        return 1;
    }
    tqo_attention(q, B, HQ, HKV, D, G64, CAP, kc, ks, kb, vc, vs, vb, lens1, attn, NULL, 0, ref);
    if (compare_out("step", out, ref, qn)) return 1;

    /* a bad argument is refused before any launch */
    if (tq_sdpa_int4_decode(&cache, d_q, HQ + 1, d_lens, max_len, attn, TQ_DEFAULT_CHUNK, ws, ws_bytes, d_out, NULL,
                            stream) == TQ_OK) {
        fprintf(stderr, "a query head count that is not a multiple of the kv heads was accepted\n");
        return 1;
    }
    printf("OK\n");
    cudaFree(ws);
    cudaFree(base);
    return 0;
}

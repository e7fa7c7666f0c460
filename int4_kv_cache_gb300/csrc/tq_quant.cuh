// tq_quant.cuh -- the group quantizer shared by the append kernel and the
// decode kernel's fused append: one group of 64 fp16 elements -> BITS-bit
// codes (BITS = 4: two per byte, element 2i in the low nibble of byte i;
// BITS = 8: one per byte) plus the group's fp16 scale and bias.
//
// Rule (the one stated in tq.h), with L = 2^BITS - 1 levels: mn, mx in fp32;
// scale = fp16(fp32(mx - mn) / L); bias = fp16(mn), with a zero minimum stored
// as +0; code = clamp(rint(fp32(x - bias) / scale), 0, L), all codes 0 when
// the scale is 0.  Every step is one IEEE fp32 operation with
// round-to-nearest-even, so the result is bit-identical to the CPU oracle.
//
// The per-element division is replaced by a multiply with fp32(1/scale):
// d * fp32(1/s) is within 3 * 2^-24 relative of fp32(d / s), so both round to
// the same integer unless a half-integer lies closer than that to the product
// (6e-6 absolute for int4, t < 32; 5e-5 for int8, t < 264): within the window
// kTieWindow of a half-integer the IEEE division decides.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace tq {

template <int BITS>
struct QuantRule {
    static constexpr float kLevels = static_cast<float>((1 << BITS) - 1);
    static constexpr float kTieWindow = BITS == 4 ? 1.0e-5f : 1.0e-4f;
};

// ---------------------------------------------- eight lanes per group of 64 --
template <int BITS>
struct GroupQ {
    uint32_t codes[BITS / 4];  // this lane's eight codes, element 0 lowest
    __half scale;
    __half bias;
};

template <int BITS = 4>
__device__ __forceinline__ GroupQ<BITS> quantize_lane8(uint4 raw) {
    using R = QuantRule<BITS>;
    float x[8];
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(h2[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        mn = fminf(mn, x[i]);
        mx = fmaxf(mx, x[i]);
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {  // the 8 lanes of a group differ in lane bits 0..2
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    if (mn == 0.0f) mn = 0.0f;  // a zero minimum is stored as +0
    const float range = __fsub_rn(mx, mn);
    GroupQ<BITS> g;
    g.scale = __float2half_rn(__fdiv_rn(range, R::kLevels));
    g.bias = __float2half_rn(mn);  // exact: mn is an fp16 value
    const float s = __half2float(g.scale);
    const float b = __half2float(g.bias);
#pragma unroll
    for (int w = 0; w < BITS / 4; ++w) g.codes[w] = 0u;
    if (s != 0.0f) {
        const float rs = __frcp_rn(s);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float d = __fsub_rn(x[i], b);  // >= 0: x >= the group minimum
            float t = __fmul_rn(d, rs);
            if (fabsf(t - floorf(t) - 0.5f) < R::kTieWindow) t = __fdiv_rn(d, s);
            int c = __float2int_rn(t);
            c = min(max(c, 0), (1 << BITS) - 1);
            g.codes[(i * BITS) / 32] |= static_cast<uint32_t>(c) << ((i * BITS) % 32);
        }
    }
    return g;
}

// ------------------------------------------------- one thread per group --
// 64 elements in eight 16-byte words -> 2 * BITS words of codes and the scale
// / bias.  No shuffles; min/max on packed fp16 pairs (exact).  Codes are
// rounded by adding 1.5 * 2^23, which leaves round-to-nearest-even(t) in the
// low bits of the fp32 sum for 0 <= t < 2^22, so no float-to-int conversion is
// needed; codes are placed with bfi.
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

template <int BITS>
__device__ __forceinline__ uint32_t code_of(float x, float b, float s, float rs) {
    using R = QuantRule<BITS>;
    const float d = __fsub_rn(x, b);  // >= 0: x >= the group minimum
    const float t = __fmul_rn(d, rs);
    float r = __fadd_rn(t, kMagic);
    if (fabsf(__fsub_rn(t, __fsub_rn(r, kMagic))) > 0.5f - R::kTieWindow) r = __fadd_rn(__fdiv_rn(d, s), kMagic);
    const uint32_t c = static_cast<uint32_t>(__float_as_int(r) - __float_as_int(kMagic));
    constexpr uint32_t L = (1u << BITS) - 1u;
    return c < L ? c : L;
}

__device__ __forceinline__ uint32_t bfi(uint32_t field, uint32_t base, uint32_t pos, uint32_t len) {
    uint32_t d;
    asm("bfi.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(field), "r"(base), "r"(pos), "r"(len));
    return d;
}

// The exact scalar rule for the codes of one 16-byte input word (8 elements;
// the rare path: a near-tie or a subnormal scale), out of line so the hot loop
// stays small.  Returns BITS / 4 words.
template <int BITS>
static __device__ __noinline__ uint2 code_word_exact(uint4 word, float b, float s, float rs) {
    const __half2* h4 = reinterpret_cast<const __half2*>(&word);
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(h4[k]);
        const int e = 2 * k;  // element within the word
        w[(e * BITS) / 32] |= code_of<BITS>(f.x, b, s, rs) << ((e * BITS) % 32);
        w[((e + 1) * BITS) / 32] |= code_of<BITS>(f.y, b, s, rs) << (((e + 1) * BITS) % 32);
    }
    return make_uint2(w[0], w[1]);
}

template <int BITS>
__device__ __forceinline__ void quantize_group64(const uint4 (&raw)[8], uint32_t (&codes)[2 * BITS], __half& scale,
                                                 __half& bias) {
    using R = QuantRule<BITS>;
    const __half2* h = reinterpret_cast<const __half2*>(raw);  // 32 pairs
    __half2 mn2 = h[0], mx2 = h[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) {
        mn2 = __hmin2(mn2, h[i]);
        mx2 = __hmax2(mx2, h[i]);
    }
    float mn = fminf(__low2float(mn2), __high2float(mn2));
    const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
    if (mn == 0.0f) mn = 0.0f;  // a zero minimum is stored as +0
    scale = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), R::kLevels));
    bias = __float2half_rn(mn);  // exact: mn is an fp16 value
    const float s = __half2float(scale), b = __half2float(bias);
#pragma unroll
    for (int j = 0; j < 2 * BITS; ++j) codes[j] = 0u;
    if (s == 0.0f) return;
    const float rs = __frcp_rn(s);
    // A normal fp16 scale is within 2^-11 of range / L, so every t stays below
    // L + 0.5 and rounds into 0..L with no clamp; subnormal scales take the
    // scalar path, which clamps.
    const bool normal = s >= 6.103515625e-05f;  // 2^-14
    const float2 nb = make_float2(-b, -b), rs2 = make_float2(rs, rs);
    const float2 mg = make_float2(kMagic, kMagic), nmg = make_float2(-kMagic, -kMagic);
    const float2 m1 = make_float2(-1.0f, -1.0f);
    // Near-tie test without per-element compares: q = e * e - c with
    // c = (0.5 - 2 * kTieWindow)^2 is one rounding of the exact value, so its
    // sign is exact, and q >= 0 for every |e| >= 0.5 - kTieWindow (and for a
    // few more, which only send their word to the exact rule).  The sign bits
    // of a word's eight q are ANDed: a clear sign bit means some q >= 0.
    constexpr float kFar = 0.5f - 2.0f * R::kTieWindow;
    const float2 nc = make_float2(-kFar * kFar, -kFar * kFar);
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // input word j: elements 8j .. 8j + 7
        uint32_t w[2] = {0u, 0u};
        uint32_t far_bits = 0x80000000u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // two elements per paired fp32 operation
            const float2 f = __half22float2(h[4 * j + k]);
            const float2 d = __fadd2_rn(f, nb);                      // x - b
            const float2 t = __fmul2_rn(d, rs2);                     // ~ d / s
            const float2 r = __fadd2_rn(t, mg);                      // rint(t) in the low bits
            const float2 e = __ffma2_rn(__fadd2_rn(r, nmg), m1, t);  // t - rint(t), exact
            const float2 q = __ffma2_rn(e, e, nc);                   // < 0 unless near a tie
            far_bits &= __float_as_uint(q.x) & __float_as_uint(q.y);
            const int p = 2 * k * BITS;  // bit position of the pair within the word(s)
            w[p / 32] = bfi(__float_as_uint(r.x), w[p / 32], p % 32, BITS);
            w[(p + BITS) / 32] = bfi(__float_as_uint(r.y), w[(p + BITS) / 32], (p + BITS) % 32, BITS);
        }
        const bool near = far_bits == 0u;
        if (near || !normal) {  // rare: redo the word with the exact scalar rule
            const uint2 x = code_word_exact<BITS>(raw[j], b, s, rs);
            w[0] = x.x;
            w[1] = x.y;
        }
        codes[j * BITS / 4] = w[0];
        if (BITS == 8) codes[j * BITS / 4 + 1] = w[1];
    }
}

}  // namespace tq

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
// The per-element division is replaced by multiplications with rounded
// reciprocals, and the IEEE division decides only where they could round to
// another code: the eight-lane quantizer tests d * fp32(1/s) (within
// 3 * 2^-24 relative of fp32(d / s)) against the window kTieWindow around a
// half-integer; the one-thread-per-group quantizer brackets fp32(d / s)
// between two products (quantize_word8).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace tq {

template <int BITS>
struct QuantRule {
    static constexpr float kLevels = static_cast<float>((1 << BITS) - 1);
    static constexpr float kTieWindow = BITS == 4 ? 1.0e-5f : 1.0e-4f;
};

// The scale and bias of a group from its minimum and maximum (fp32 values of
// fp16 elements) and the sign bit of its first element: the stored scale is
// fp16(fp32(max - min) / L) with a zero minimum taken as +0.  The rule's
// maximum is the first element holding the largest value, so in a group of
// zeros the range is (first element) - (+0): -0 when the group opens with -0
// (the scale is then -0), +0 otherwise.
template <int BITS>
__device__ __forceinline__ void group_scale_bias(float mn, float mx, bool first_neg, __half& scale, __half& bias) {
    using R = QuantRule<BITS>;
    if (mn == 0.0f) mn = 0.0f;  // a zero minimum is stored as +0
    if (mx == 0.0f) mx = first_neg && mn == 0.0f ? -0.0f : 0.0f;
    scale = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), R::kLevels));
    bias = __float2half_rn(mn);  // exact: mn is an fp16 value
}

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
    // the group's first element sits in the lowest of its eight lanes
    const uint32_t first = __shfl_sync(0xffffffffu, raw.x, (threadIdx.x & 31) & ~7);
    GroupQ<BITS> g;
    group_scale_bias<BITS>(mn, mx, (first & 0x8000u) != 0u, g.scale, g.bias);
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

// fp32(x) + c and fp32(x) - c with one rounding each, x an fp16 value (widened
// exactly).
__device__ __forceinline__ float add_h_f(__half x, float c) {
    float d;
    asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(__half_as_ushort(x)), "f"(c));
    return d;
}
__device__ __forceinline__ float sub_h_f(__half x, float c) {
    float d;
    asm("sub.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(__half_as_ushort(x)), "f"(c));
    return d;
}

// Multipliers bracketing 1 / s: lo <= (1 / s)(1 - 2^-23) and
// hi >= (1 / s)(1 + 2^-23).  rs = fp32(1 / s) is within 2^-24 relative of
// 1 / s and each product below adds at most 2^-24 more, so a relative step of
// 2^-21 keeps both bounds.
struct RecipBracket {
    float lo, hi;
};
__device__ __forceinline__ RecipBracket recip_bracket(float rs) {
    return {__fmul_rn(rs, 1.0f - 0x1p-21f), __fmul_rn(rs, 1.0f + 0x1p-21f)};
}

// The codes of one 16-byte word (8 elements, element 0 lowest; BITS / 4
// words) of a group with scale s > 0, bias b, rs = fp32(1 / s) and the
// bracket br of 1 / s.  For d = fp32(x - b) >= 0, fp32(d / s) is within
// 2^-24 relative of d / s, so it lies in [d * br.lo, d * br.hi]; rint is
// non-decreasing, so where rint(d * br.lo) == rint(d * br.hi) that is also
// rint(fp32(d / s)), the code.  Each rint is one fused multiply-add with
// 1.5 * 2^23, which leaves round-to-nearest-even of the exact product in the
// low bits.  A normal fp16 scale is within 2^-11 of range / L, so every
// product stays below L + 0.5 and no clamp is needed.  A word where the two
// roundings differ for some element (a half-integer lies in its interval:
// within about 2^-22 relative of a tie) or whose scale is subnormal takes the
// exact scalar rule.
template <int BITS>
__device__ __forceinline__ uint2 quantize_word8(const uint4& raw, float b, float s, float rs, RecipBracket br) {
    const bool normal = s >= 6.103515625e-05f;  // 2^-14
    const float2 lo2 = make_float2(br.lo, br.lo), hi2 = make_float2(br.hi, br.hi);
    const float2 mg = make_float2(kMagic, kMagic);
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
    // The code bits of an element are the low bits of its fp32 result (the
    // bits of 1.5 * 2^23 are zero below bit 22), so the word is put together
    // by a tree of bit-field inserts: pairs, then quads, then the word.
    uint32_t pr[4], t[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // two elements per paired fp32 operation
        const float2 d = make_float2(sub_h_f(__low2half(h[k]), b), sub_h_f(__high2half(h[k]), b));  // x - b
        const float2 ra = __ffma2_rn(d, lo2, mg), rb = __ffma2_rn(d, hi2, mg);
        t[k] = (__float_as_uint(ra.x) ^ __float_as_uint(rb.x)) | (__float_as_uint(ra.y) ^ __float_as_uint(rb.y));
        pr[k] = bfi(__float_as_uint(ra.y), __float_as_uint(ra.x), BITS, BITS);  // elements 2k, 2k + 1
    }
    const uint32_t diff = (t[0] | t[1]) | (t[2] | t[3]);
    uint2 w;
    if (BITS == 4) {
        w.x = bfi(bfi(pr[3], pr[2], 8, 8), bfi(pr[1], pr[0], 8, 8), 16, 16);
        w.y = 0u;
    } else {
        w.x = bfi(pr[1], pr[0], 16, 16);
        w.y = bfi(pr[3], pr[2], 16, 16);
    }
    if (diff != 0u || !normal) return code_word_exact<BITS>(raw, b, s, rs);  // rare: the exact scalar rule
    return w;
}

template <int BITS>
__device__ __forceinline__ void quantize_group64(const uint4 (&raw)[8], uint32_t (&codes)[2 * BITS], __half& scale,
                                                 __half& bias) {
    const __half2* h = reinterpret_cast<const __half2*>(raw);  // 32 pairs
    __half2 mn2 = h[0], mx2 = h[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) {
        mn2 = __hmin2(mn2, h[i]);
        mx2 = __hmax2(mx2, h[i]);
    }
    const float mn = fminf(__low2float(mn2), __high2float(mn2));
    const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
    group_scale_bias<BITS>(mn, mx, (raw[0].x & 0x8000u) != 0u, scale, bias);
    const float s = __half2float(scale), b = __half2float(bias);
#pragma unroll
    for (int j = 0; j < 2 * BITS; ++j) codes[j] = 0u;
    if (s == 0.0f) return;
    const float rs = __frcp_rn(s);
    const RecipBracket br = recip_bracket(rs);
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // input word j: elements 8j .. 8j + 7
        const uint2 x = quantize_word8<BITS>(raw[j], b, s, rs, br);
        codes[j * BITS / 4] = x.x;
        if (BITS == 8) codes[j * BITS / 4 + 1] = x.y;
    }
}

}  // namespace tq

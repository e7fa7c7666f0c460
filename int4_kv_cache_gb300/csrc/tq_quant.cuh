// tq_quant.cuh -- the group quantizer shared by the append kernel and the
// decode kernel's fused append: one group of 64 fp16 elements held by eight
// consecutive lanes (eight elements each) -> eight 4-bit codes per lane plus the
// group's fp16 scale and bias.
//
// Rule (the one stated in tq.h): mn, mx in fp32; scale = fp16(fp32(mx - mn) /
// 15); bias = fp16(mn), with a zero minimum stored as +0; code =
// clamp(rint(fp32(x - bias) / scale), 0, 15), all codes 0 when the scale is 0.
// Every step is one IEEE fp32 operation with round-to-nearest-even, so the
// result is bit-identical to the CPU oracle.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace tq {

struct GroupQ {
    uint32_t codes;  // eight 4-bit codes, element 0 in bits 0..3
    __half scale;
    __half bias;
};

__device__ __forceinline__ GroupQ quantize_lane8(uint4 raw) {
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
    GroupQ g;
    g.scale = __float2half_rn(__fdiv_rn(range, 15.0f));
    g.bias = __float2half_rn(mn);  // exact: mn is an fp16 value
    const float s = __half2float(g.scale);
    const float b = __half2float(g.bias);
    uint32_t codes = 0;
    if (s != 0.0f) {
        // t = fp32(d / s) is rounded to an integer.  d * fp32(1/s) is within
        // 2^-22 relative (< 4e-6 absolute, as t <= 15.01) of that quotient, so
        // both round to the same integer unless a half-integer lies within 4e-6
        // of the product: only then is the IEEE division itself evaluated.
        const float rs = __frcp_rn(s);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float d = __fsub_rn(x[i], b);  // >= 0: x >= the group minimum
            float t = __fmul_rn(d, rs);
            if (fabsf(t - floorf(t) - 0.5f) < 1.0e-5f) t = __fdiv_rn(d, s);
            int c = __float2int_rn(t);
            c = min(max(c, 0), 15);
            codes |= static_cast<uint32_t>(c) << (4 * i);
        }
    }
    g.codes = codes;
    return g;
}

// The same rule with one thread per group: 64 elements in eight 16-byte
// words -> eight 32-bit words of codes (element 2i in the low nibble of byte
// i) and the scale / bias bits.  No shuffles; min/max on packed fp16 pairs
// (exact).  Codes are rounded by adding 1.5 * 2^23, which leaves
// round-to-nearest-even(t) in the low bits of the fp32 sum for 0 <= t < 2^22
// (t < 32 here), so no float-to-int conversion is needed.
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

// d * fp32(1/s) is within 3 * 2^-24 relative (< 6e-6 absolute, t < 32) of
// fp32(d / s), so both round to the same integer unless a half-integer lies
// within 1e-5 of t: only then is the IEEE division evaluated.
__device__ __forceinline__ uint32_t code_of(float x, float b, float s, float rs) {
    const float d = __fsub_rn(x, b);  // >= 0: x >= the group minimum
    const float t = __fmul_rn(d, rs);
    float r = __fadd_rn(t, kMagic);
    if (fabsf(__fsub_rn(t, __fsub_rn(r, kMagic))) > 0.49999f) r = __fadd_rn(__fdiv_rn(d, s), kMagic);
    const uint32_t c = static_cast<uint32_t>(__float_as_int(r) - __float_as_int(kMagic));
    return c < 15u ? c : 15u;
}

// The exact scalar rule for one word of 8 codes (the rare path: a near-tie
// or a subnormal scale); kept out of line so the hot loop stays small.
static __device__ __noinline__ uint32_t code_word_exact(uint4 word, float b, float s, float rs) {
    const __half2* h4 = reinterpret_cast<const __half2*>(&word);
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(h4[k]);
        w |= (code_of(f.x, b, s, rs) | (code_of(f.y, b, s, rs) << 4)) << (8 * k);
    }
    return w;
}

__device__ __forceinline__ uint32_t bfi4(uint32_t field, uint32_t base, uint32_t pos) {
    uint32_t d;
    asm("bfi.b32 %0, %1, %2, %3, 4;" : "=r"(d) : "r"(field), "r"(base), "r"(pos));
    return d;
}

__device__ __forceinline__ void quantize_group64(const uint4 (&raw)[8], uint32_t (&codes)[8], __half& scale,
                                                 __half& bias) {
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
    scale = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
    bias = __float2half_rn(mn);  // exact: mn is an fp16 value
    const float s = __half2float(scale), b = __half2float(bias);
    if (s == 0.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) codes[j] = 0u;
        return;
    }
    const float rs = __frcp_rn(s);
    // A normal fp16 scale is within 2^-11 of range / 15, so every t stays below
    // 15.01 and rounds into 0..15 with no clamp; subnormal scales take the
    // scalar path, which clamps.
    const bool normal = s >= 6.103515625e-05f;  // 2^-14
    const float2 nb = make_float2(-b, -b), rs2 = make_float2(rs, rs);
    const float2 mg = make_float2(kMagic, kMagic), nmg = make_float2(-kMagic, -kMagic);
    const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t w = 0;
        bool near = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // elements 8j + 2k, 8j + 2k + 1: two per paired fp32 operation
            const float2 f = __half22float2(h[4 * j + k]);
            const float2 d = __fadd2_rn(f, nb);       // x - b
            const float2 t = __fmul2_rn(d, rs2);      // ~ d / s
            const float2 r = __fadd2_rn(t, mg);       // rint(t) in the low bits
            const float2 e = __ffma2_rn(__fadd2_rn(r, nmg), m1, t);  // t - rint(t), exact
            near |= (fabsf(e.x) > 0.49999f) | (fabsf(e.y) > 0.49999f);
            w = bfi4(__float_as_uint(r.x), w, 8 * k);
            w = bfi4(__float_as_uint(r.y), w, 8 * k + 4);
        }
        if (near || !normal) w = code_word_exact(raw[j], b, s, rs);  // rare
        codes[j] = w;
    }
}

}  // namespace tq

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

}  // namespace tq

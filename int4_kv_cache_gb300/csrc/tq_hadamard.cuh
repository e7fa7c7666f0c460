// tq_hadamard.cuh -- the normalised Sylvester Hadamard rotation across one
// warp ("Running and Evaluating TurboQuant optimized Gemma 4", TurboQuant
// section: H / sqrt(n) spreads an outlier over every coordinate before
// quantisation and is its own inverse).
//
// A row of n = 32 * E values; lane l holds elements E * l .. E * l + E - 1.
// Fast transform in fp32 with the stages in increasing order h = 1, 2, ...,
// n/2: each pair (i, i + h) with bit h of i clear becomes (x_i + x_{i+h},
// x_i - x_{i+h}).  Stages h < E stay inside a lane; stage h >= E pairs lane l
// with lane l ^ (h / E).  Then every value is multiplied by `scale` (the fp32
// value nearest 1/sqrt(n)).  The same operations in the same order as a plain
// sequential transform, so the fp32 results are identical to it.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace tq {

template <int E>
__device__ __forceinline__ void hadamard_warp(float (&v)[E], int lane, float scale) {
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int i = 0; i < E; ++i) {
            if ((i & h) == 0) {
                const float u = v[i], w = v[i + h];
                v[i] = __fadd_rn(u, w);
                v[i + h] = __fsub_rn(u, w);
            }
        }
    }
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1) {
        const bool upper = (lane & hl) != 0;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, v[i], hl);
            v[i] = upper ? __fsub_rn(other, v[i]) : __fadd_rn(v[i], other);
        }
    }
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = __fmul_rn(v[i], scale);
}

// Building blocks for rows spread over a few lanes in other layouts (the
// decode kernel's query fragments and fused append): the stages h < E inside
// a lane's E consecutive elements, and one stage whose pairs sit in lanes
// lane and lane ^ hl (the lane with bit hl set holds the upper element).
// Called in increasing h, they perform the butterflies of the sequential
// transform with the same round-to-nearest operations.
template <int E>
__device__ __forceinline__ void hadamard_in_lane(float (&v)[E]) {
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int i = 0; i < E; ++i) {
            if ((i & h) == 0) {
                const float u = v[i], w = v[i + h];
                v[i] = __fadd_rn(u, w);
                v[i + h] = __fsub_rn(u, w);
            }
        }
    }
}

template <int E>
__device__ __forceinline__ void hadamard_across_lanes(float (&v)[E], int lane, int hl) {
    const bool upper = (lane & hl) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const float other = __shfl_xor_sync(0xffffffffu, v[i], hl);
        v[i] = upper ? __fsub_rn(other, v[i]) : __fadd_rn(v[i], other);
    }
}

// E consecutive fp16 values <-> floats (E = 2, 4, 8: 4, 8 or 16 bytes).
template <int E>
__device__ __forceinline__ void halves_to_floats(const void* src, float (&v)[E]) {
    const __half2* h = reinterpret_cast<const __half2*>(src);
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        const float2 f = __half22float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

template <int E>
__device__ __forceinline__ void floats_to_halves(const float (&v)[E], void* dst) {
    __half2* h = reinterpret_cast<__half2*>(dst);
#pragma unroll
    for (int i = 0; i < E / 2; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
}

}  // namespace tq

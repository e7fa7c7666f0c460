// dequant.cu -- expands the int4 cache into fp16 K and V: the float cache that
// a dequantize-then-attend decode builds before running ordinary SDPA ("Fused
// int4 Attention for Gemma 4 31B on Apple Silicon", What I Built Instead: the
// path the fused kernel replaces).  It exists as the comparison point for the
// fused decode, not as part of it.
//
// value = fp16_rne(fp32(scale * code + bias)): the product is exact in fp32
// (11 x 4 significant bits), so one fused multiply-add rounds once to fp32,
// then the conversion rounds to binary16.
//
// Work split: one thread per 8 elements (one 32-bit word of codes, 16 bytes of
// output), grid-stride over [B][Hkv][n_rows][D/8] for K (blockIdx.y = 0) and
// V (blockIdx.y = 1); every store is a 16-byte coalesced write.
#include <cuda_fp16.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

template <int BITS>
__global__ void __launch_bounds__(256) dequant_kernel(const DequantParams p) {
    const int kv = blockIdx.y;
    const uint8_t* codes = kv ? p.v_codes : p.k_codes;
    const uint16_t* scale = kv ? p.v_scale : p.k_scale;
    const uint16_t* bias = kv ? p.v_bias : p.k_bias;
    uint16_t* out = kv ? p.v_out : p.k_out;
    const int words = p.head_dim / 8;  // 8 codes per thread: one 32-bit word (int4) or two (int8)
    const int ng = p.head_dim / kGroup;
    const long long total = static_cast<long long>(p.batch) * p.num_kv_heads * p.n_rows * words;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = i / words;  // over [B][Hkv][n_rows]
        const int w = static_cast<int>(i - row * words);
        const long long bh = row / p.n_rows;
        const long long src = bh * p.capacity + (row - bh * p.n_rows);
        const uint8_t* cp = codes + src * (p.head_dim * BITS / 8) + w * BITS;  // this thread's 8 codes
        uint32_t c[2];
        if constexpr (BITS == 8) {
            const uint2 v = __ldcs(reinterpret_cast<const uint2*>(cp));
            c[0] = v.x;
            c[1] = v.y;
        } else {
            c[0] = __ldcs(reinterpret_cast<const uint32_t*>(cp));
            c[1] = 0u;
        }
        const int g = (w * 8) / kGroup;
        const float s = __half2float(__ushort_as_half(__ldg(scale + src * ng + g)));
        const float b = __half2float(__ushort_as_half(__ldg(bias + src * ng + g)));
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t n0, n1;  // codes of elements 2j, 2j + 1
            if constexpr (BITS == 8) {
                n0 = (c[j / 2] >> (16 * (j % 2))) & 0xFFu;
                n1 = (c[j / 2] >> (16 * (j % 2) + 8)) & 0xFFu;
            } else {
                n0 = (c[0] >> (8 * j)) & 0xFu;
                n1 = (c[0] >> (8 * j + 4)) & 0xFu;
            }
            const float lo = __fmaf_rn(s, static_cast<float>(n0), b);
            const float hi = __fmaf_rn(s, static_cast<float>(n1), b);
            h[j] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
                   (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
        }
        __stcs(reinterpret_cast<uint4*>(out + row * p.head_dim) + w, make_uint4(h[0], h[1], h[2], h[3]));
    }
}

}  // namespace

cudaError_t launch_dequant(const DequantParams& p, int sm_count, cudaStream_t stream) {
    const long long total = static_cast<long long>(p.batch) * p.num_kv_heads * p.n_rows * (p.head_dim / 8);
    if (total == 0) return cudaSuccess;
    const long long want = (total + 255) / 256;
    const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 152) * 8;
    const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
    if (p.bits == 8) dequant_kernel<8><<<dim3(blocks, 2), 256, 0, stream>>>(p);
    else dequant_kernel<4><<<dim3(blocks, 2), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace tq

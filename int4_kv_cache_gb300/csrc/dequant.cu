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
// Work split: one thread per 8 elements (one 32-bit word of codes, 16 bytes
// of output); a CTA of 256 threads covers 256 / (D / 8) consecutive rows of one
// (sequence, kv head) per pass, blockIdx.z selects the (sequence, kv head) and
// blockIdx.y K or V, so no 64-bit division is left in the loop; every store is
// a 16-byte coalesced write.
#include <cuda_fp16.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

template <int BITS, int D>
__global__ void __launch_bounds__(256) dequant_kernel(const DequantParams p) {
    constexpr int kWords = D / 8;               // threads per row: 8 codes each
    constexpr int kRows = 256 / kWords;         // rows per CTA pass
    constexpr int kNg = D / kGroup;
    const int kv = blockIdx.y;
    const long long bh = blockIdx.z;            // (sequence, kv head)
    const uint8_t* codes = (kv ? p.v_codes : p.k_codes) + bh * p.capacity * (D * BITS / 8);
    const uint16_t* scale = (kv ? p.v_scale : p.k_scale) + bh * p.capacity * kNg;
    const uint16_t* bias = (kv ? p.v_bias : p.k_bias) + bh * p.capacity * kNg;
    uint16_t* out = (kv ? p.v_out : p.k_out) + bh * p.n_rows * D;
    const int w = threadIdx.x % kWords;
    const int g = (w * 8) / kGroup;
    for (int r = blockIdx.x * kRows + threadIdx.x / kWords; r < p.n_rows; r += gridDim.x * kRows) {
        const uint8_t* cp = codes + static_cast<long long>(r) * (D * BITS / 8) + w * BITS;  // this thread's 8 codes
        uint32_t c[2];
        if constexpr (BITS == 8) {
            const uint2 v = __ldcs(reinterpret_cast<const uint2*>(cp));
            c[0] = v.x;
            c[1] = v.y;
        } else {
            c[0] = __ldcs(reinterpret_cast<const uint32_t*>(cp));
            c[1] = 0u;
        }
        const float s = __half2float(__ushort_as_half(__ldg(scale + static_cast<long long>(r) * kNg + g)));
        const float b = __half2float(__ushort_as_half(__ldg(bias + static_cast<long long>(r) * kNg + g)));
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
        __stcs(reinterpret_cast<uint4*>(out + static_cast<long long>(r) * D) + w, make_uint4(h[0], h[1], h[2], h[3]));
    }
}

template <int BITS, int D>
cudaError_t launch_dq(const DequantParams& p, int sm_count, cudaStream_t stream) {
    constexpr int kRows = 256 / (D / 8);
    const long long heads = static_cast<long long>(p.batch) * p.num_kv_heads;
    if (heads > 65535) return cudaErrorInvalidConfiguration;
    // about eight CTAs per SM in all, each (sequence, kv head) slice strided over its rows
    const long long per_head = (static_cast<long long>(sm_count > 0 ? sm_count : 152) * 8 + 2 * heads - 1) / (2 * heads);
    const long long need = (p.n_rows + kRows - 1) / kRows;
    const unsigned x = static_cast<unsigned>(per_head < need ? (per_head > 0 ? per_head : 1) : need);
    dequant_kernel<BITS, D><<<dim3(x, 2, static_cast<unsigned>(heads)), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequant(const DequantParams& p, int sm_count, cudaStream_t stream) {
    if (p.n_rows == 0 || p.batch == 0 || p.num_kv_heads == 0) return cudaSuccess;
    const bool i8 = p.bits == 8;
    switch (p.head_dim) {
        case 64: return i8 ? launch_dq<8, 64>(p, sm_count, stream) : launch_dq<4, 64>(p, sm_count, stream);
        case 128: return i8 ? launch_dq<8, 128>(p, sm_count, stream) : launch_dq<4, 128>(p, sm_count, stream);
        case 256: return i8 ? launch_dq<8, 256>(p, sm_count, stream) : launch_dq<4, 256>(p, sm_count, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tq

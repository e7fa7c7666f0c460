// quantize.cu -- quantize-on-store: fp16 K/V rows -> packed int4 codes plus
// fp16 scale/bias per group of 64, written in place into the cache.
//
// Method: "turboquant-llama3.170B" README, decode-step listing (quantize K,V to
// int4 after RoPE, then store) and the Gemma page, Background (MLX-style int4
// with a per-group scale and bias).  The rounding rule is the one stated in
// tq.h; every step is a single IEEE fp32 operation with round-to-nearest-even,
// so codes, scales and biases are bit-identical to the CPU oracle.  The
// per-element division is replaced by a multiply with the reciprocal wherever
// that provably rounds to the same code (tq_quant.cuh).
//
// Work split: one thread per (row, group of 64): it loads the group of K and
// the group of V (eight 16-byte words each, all issued before any use), and
// writes 32 bytes of codes per tensor and the four scale / bias halves.  With
// no cross-lane reductions the per-group work (min/max, the scale division,
// the reciprocal) is spread over 64 elements.
#include "tq_device.cuh"
#include "tq_hadamard.cuh"
#include "tq_internal.h"
#include "tq_quant.cuh"

namespace tq {

namespace {

constexpr int kQuantThreads = 128;

// Rotate the rows held in one warp's staging tile in place (32 groups = 32 /
// ng whole rows): lane l takes elements E*l .. E*l+E-1 of each row in turn.
template <int E>
__device__ __forceinline__ void rotate_staged(uint4 (&tile)[32][8], int lane, int ng, float scale) {
    const int d = E * lane;
    for (int rr = 0; rr < 32 / ng; ++rr) {
        const int r = rr * ng + d / kGroup, w = (d % kGroup) / 8;
        uint16_t* ptr = reinterpret_cast<uint16_t*>(&tile[r][w ^ (r & 7)]) + (d % 8);
        float v[E];
        halves_to_floats<E>(ptr, v);
        hadamard_warp<E>(v, lane, scale);
        floats_to_halves<E>(v, ptr);
    }
}

template <int BITS>
__global__ void __launch_bounds__(kQuantThreads) quantize_append_kernel(const AppendParams p) {
    // staging: per warp and tensor, 32 groups x 8 words of 16 bytes; word w of
    // group r sits at slot w ^ (r & 7), so that the eight lanes of each phase of
    // a 16-byte shared access hit eight different bank groups
    __shared__ uint4 stage[kQuantThreads / 32][2][32][8];
    pdl_launch_dependents();  // no effect unless the next launch is a programmatic dependent
    const int ng = p.head_dim / kGroup;
    const long long n_groups = static_cast<long long>(p.batch) * p.num_kv_heads * p.n_new * ng;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long warp_base = static_cast<long long>(blockIdx.x) * kQuantThreads + warp * 32;
    if (warp_base >= n_groups) return;  // the whole warp

    // coalesced loads of the warp's 32 consecutive groups (4 KB per tensor:
    // group gi starts at element gi * 64 of k_new / v_new)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const uint4* src = reinterpret_cast<const uint4*>(t ? p.v_new : p.k_new) + warp_base * 8;
        uint4 w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + (lane >> 3);  // group within the warp's 32
            w[j] = warp_base + r < n_groups ? __ldcs(src + 32 * j + lane) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + (lane >> 3), word = lane & 7;
            stage[warp][t][r][word ^ (r & 7)] = w[j];
        }
    }
    __syncwarp();
    if (p.flags & (TQ_ROTATE_K | TQ_ROTATE_V)) {  // the same for the whole launch
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
            if (!(p.flags & (t ? TQ_ROTATE_V : TQ_ROTATE_K))) continue;
            switch (p.head_dim) {
                case 64: rotate_staged<2>(stage[warp][t], lane, ng, p.rot_scale); break;
                case 128: rotate_staged<4>(stage[warp][t], lane, ng, p.rot_scale); break;
                default: rotate_staged<8>(stage[warp][t], lane, ng, p.rot_scale); break;
            }
        }
        __syncwarp();
    }

    const long long gi = warp_base + lane;
    if (gi >= n_groups) return;
    const int g = static_cast<int>(gi % ng);
    const long long row = gi / ng;  // over [B][Hkv][n_new]
    const int i = static_cast<int>(row % p.n_new);
    const long long bh = row / p.n_new;  // b * Hkv + h
    const int b = static_cast<int>(bh / p.num_kv_heads);
    const int wp = __ldg(p.write_pos + b);
    if (wp < 0 || static_cast<long long>(wp) + p.n_new > p.capacity) {
        if (p.status != nullptr && g == 0 && i == 0) atomicOr(p.status, TQ_DEV_WRITE_POS);
        return;
    }
    const long long dst_row =
        kv_row(p.map, p.num_kv_heads, b, static_cast<int>(bh - static_cast<long long>(b) * p.num_kv_heads), wp + i,
               p.status);
    const long long code_off = dst_row * (p.head_dim * BITS / 8) + g * (kGroup * BITS / 8);  // 32-byte aligned
    const long long sb = dst_row * ng + g;
#pragma unroll 1
    for (int t = 0; t < 2; ++t) {
        uint4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = stage[warp][t][lane][j ^ (lane & 7)];
        uint32_t c[2 * BITS];
        __half sc, bi;
        quantize_group64<BITS>(x, c, sc, bi);
        uint4* dst = reinterpret_cast<uint4*>((t ? p.v_codes : p.k_codes) + code_off);
#pragma unroll
        for (int w = 0; w < BITS / 2; ++w) dst[w] = make_uint4(c[4 * w], c[4 * w + 1], c[4 * w + 2], c[4 * w + 3]);
        (t ? p.v_scale : p.k_scale)[sb] = __half_as_ushort(sc);
        (t ? p.v_bias : p.k_bias)[sb] = __half_as_ushort(bi);
    }
}

}  // namespace

cudaError_t launch_quantize_append(const AppendParams& p, cudaStream_t stream) {
    const long long groups = static_cast<long long>(p.batch) * p.num_kv_heads * p.n_new * (p.head_dim / kGroup);
    const int block = kQuantThreads;
    const long long blocks = (groups + block - 1) / block;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (p.bits == 8) quantize_append_kernel<8><<<static_cast<unsigned>(blocks), block, 0, stream>>>(p);
    else quantize_append_kernel<4><<<static_cast<unsigned>(blocks), block, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_quantize_append_primary(const AppendParams& p, cudaStream_t stream) {
    return launch_quantize_append(p, stream);
}

}  // namespace tq

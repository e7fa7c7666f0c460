// quantize.cu -- quantize-on-store: fp16 K/V rows -> packed int4 codes plus
// fp16 scale/bias per group of 64, written in place into the cache.
//
// Method: "turboquant-llama3.170B" README, decode-step listing (quantize K,V to
// int4 after RoPE, then store) and the Gemma page, Background (MLX-style int4
// with a per-group scale and bias).  The rounding rule is the one stated in
// tq.h; every step is a single IEEE fp32 operation with round-to-nearest-even
// (__fsub_rn / __fdiv_rn / __float2int_rn), so codes, scales and biases are
// bit-identical to the CPU oracle.  The per-element division is replaced by a
// multiply with the reciprocal wherever that provably rounds to the same code.
//
// Work split: eight lanes own one group of 64 elements (16 bytes = 8 halves
// each), which makes every global access a 16-byte (input) or 4-byte (codes)
// coalesced transaction; min/max are reduced with three xor-shuffles.
#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_quant.cuh"

namespace tq {

namespace {

__global__ void __launch_bounds__(256) quantize_append_kernel(const AppendParams p) {
    pdl_launch_dependents();  // no effect unless the next launch is a programmatic dependent
    const int ng = p.head_dim / kGroup;
    const long long n_groups = static_cast<long long>(p.batch) * p.num_kv_heads * p.n_new * ng;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int part = static_cast<int>(tid & 7);
    const long long gidx = tid >> 3;
    const bool valid = gidx < n_groups;  // whole groups of 8 lanes agree
    const long long gi = valid ? gidx : 0;
    const int g = static_cast<int>(gi % ng);
    const long long row = gi / ng;  // over [B][Hkv][n_new]
    const int i = static_cast<int>(row % p.n_new);
    const long long bh = row / p.n_new;  // b * Hkv + h
    const int b = static_cast<int>(bh / p.num_kv_heads);

    const long long src = row * p.head_dim + g * kGroup + part * 8;  // in halves
    uint4 kr = make_uint4(0, 0, 0, 0), vr = make_uint4(0, 0, 0, 0);
    int wp = 0;
    if (valid) {
        kr = __ldcs(reinterpret_cast<const uint4*>(p.k_new + src));
        vr = __ldcs(reinterpret_cast<const uint4*>(p.v_new + src));
        wp = __ldg(p.write_pos + b);
    }
    const GroupQ kq = quantize_lane8(kr);  // every lane takes part in the shuffles
    const GroupQ vq = quantize_lane8(vr);
    if (!valid) return;

    const bool pos_ok = wp >= 0 && static_cast<long long>(wp) + p.n_new <= p.capacity;
    if (!pos_ok) {
        if (p.status != nullptr && part == 0 && g == 0 && i == 0) atomicOr(p.status, TQ_DEV_WRITE_POS);
        return;
    }
    const long long dst_row = bh * p.capacity + wp + i;
    const long long code_off = dst_row * (p.head_dim / 2) + g * (kGroup / 2) + part * 4;
    *reinterpret_cast<uint32_t*>(p.k_codes + code_off) = kq.codes;
    *reinterpret_cast<uint32_t*>(p.v_codes + code_off) = vq.codes;
    if (part == 0) {
        const long long sb = dst_row * ng + g;
        p.k_scale[sb] = __half_as_ushort(kq.scale);
        p.k_bias[sb] = __half_as_ushort(kq.bias);
        p.v_scale[sb] = __half_as_ushort(vq.scale);
        p.v_bias[sb] = __half_as_ushort(vq.bias);
    }
}

}  // namespace

cudaError_t launch_quantize_append(const AppendParams& p, cudaStream_t stream) {
    const long long groups = static_cast<long long>(p.batch) * p.num_kv_heads * p.n_new * (p.head_dim / kGroup);
    const long long threads = groups * 8;
    const int block = 256;
    const long long blocks = (threads + block - 1) / block;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    quantize_append_kernel<<<static_cast<unsigned>(blocks), block, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_quantize_append_primary(const AppendParams& p, cudaStream_t stream) {
    return launch_quantize_append(p, stream);
}

}  // namespace tq

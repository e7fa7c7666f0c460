// decode_simt.cu -- split-K phase 1 of int4 decode attention on CUDA cores.
//
// This is the plain fp32-FMA formulation, kept as the comparison point for
// the tensor-core kernel: per token it dequantises K and V in registers
// (value = scale * code + bias, "Fused int4 Attention for Gemma 4 31B",
// What I Built Instead) and runs the online softmax of the
// "turboquant-llama3.170B" README (kernel paragraph), one CTA per
// (run of chunks, kv head, sequence) as in its split-K paragraph.
//
// CTA = 128 threads.  Per tile of 64 tokens:
//   scores: thread pair (token, half of head_dim) -> G partial dots, one shuffle
//   softmax: tile max / sum per head through shared memory
//   P.V:    thread owns head_dim element(s) tid (+128) for all G heads
#include <math.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kSimtThreads = 128;
constexpr int kSimtTile = kSimtTileTokens;
constexpr int kGMax = 8;

__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b) {
    int len = __ldg(p.seq_lens + b);
    if (len < 0 || len > p.max_seq_len) {
        if (p.status != nullptr && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            atomicOr(p.status, TQ_DEV_SEQ_LEN);
        len = min(max(len, 0), p.max_seq_len);
    }
    return len;
}

template <int D>
__global__ void __launch_bounds__(kSimtThreads) decode_simt_kernel(const DecodeParams p) {
    constexpr int NG = D / kGroup;
    constexpr int HALF = D / 2;  // elements per half row
    constexpr int DPT = (D + kSimtThreads - 1) / kSimtThreads;
    __shared__ float q_s[kGMax][D];
    __shared__ float p_s[kSimtTile][kGMax];
    __shared__ float red_max[kSimtThreads / 32][kGMax];
    __shared__ float red_sum[kSimtThreads / 32][kGMax];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int G = p.group_q;
    const int len = clamp_len(p, b);
    const int t_begin = run_begin(split, p.units, p.n_splits, p.unit_tokens);
    const int t_end = min(run_begin(split + 1, p.units, p.n_splits, p.unit_tokens), len);

    pdl_launch_dependents();

    for (int idx = tid; idx < kGMax * D; idx += kSimtThreads) {
        const int h = idx / D, d = idx % D;
        q_s[h][d] = h < G ? __half2float(__ushort_as_half(
                                p.q[(static_cast<long long>(b) * p.num_q_heads + kvh * G + h) * D + d]))
                          : 0.0f;
    }
    __syncthreads();

    float m_run[kGMax], l_run[kGMax], acc[kGMax][DPT];
#pragma unroll
    for (int h = 0; h < kGMax; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.0f;
#pragma unroll
        for (int j = 0; j < DPT; ++j) acc[h][j] = 0.0f;
    }
    const long long row0 = (static_cast<long long>(b) * p.num_kv_heads + kvh) * p.capacity;

    for (int t0 = t_begin; t0 < t_end; t0 += kSimtTile) {
        // ---- scores: thread pair per token
        const int tok = tid >> 1, hf = tid & 1;
        const int t = t0 + tok;
        float sc[kGMax];
#pragma unroll
        for (int h = 0; h < kGMax; ++h) sc[h] = 0.0f;
        if (t < t_end) {
            const uint8_t* kc = p.k_codes + (row0 + t) * (D / 2) + hf * (HALF / 2);
            const uint16_t* ks = p.k_scale + (row0 + t) * NG;
            const uint16_t* kb = p.k_bias + (row0 + t) * NG;
            for (int j = 0; j < HALF / 2; ++j) {
                const int d0 = hf * HALF + 2 * j;
                const int g = d0 / kGroup;
                const float s = __half2float(__ushort_as_half(ks[g]));
                const float bb = __half2float(__ushort_as_half(kb[g]));
                const uint8_t byte = kc[j];
                const float k0 = fmaf(s, static_cast<float>(byte & 0xf), bb);
                const float k1 = fmaf(s, static_cast<float>(byte >> 4), bb);
#pragma unroll
                for (int h = 0; h < kGMax; ++h) sc[h] = fmaf(q_s[h][d0 + 1], k1, fmaf(q_s[h][d0], k0, sc[h]));
            }
        }
        float tmax[kGMax];
#pragma unroll
        for (int h = 0; h < kGMax; ++h) {
            sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], 1);
            sc[h] = (t < t_end) ? sc[h] * p.score_scale_log2 : -INFINITY;
            float v = sc[h];
#pragma unroll
            for (int off = 2; off < 32; off <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
            tmax[h] = v;
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < kGMax; ++h) red_max[warp][h] = tmax[h];
        }
        __syncthreads();
        float mnew[kGMax], muse[kGMax], alpha[kGMax];
#pragma unroll
        for (int h = 0; h < kGMax; ++h) {
            float v = red_max[0][h];
#pragma unroll
            for (int w = 1; w < kSimtThreads / 32; ++w) v = fmaxf(v, red_max[w][h]);
            mnew[h] = fmaxf(m_run[h], v);
            muse[h] = mnew[h] == -INFINITY ? 0.0f : mnew[h];
            alpha[h] = m_run[h] == -INFINITY ? 0.0f : exp2f(m_run[h] - muse[h]);
        }
        float psum[kGMax];
#pragma unroll
        for (int h = 0; h < kGMax; ++h) {
            const float pr = (t < t_end) ? exp2f(sc[h] - muse[h]) : 0.0f;
            if (hf == 0) p_s[tok][h] = pr;
            float v = hf == 0 ? pr : 0.0f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            psum[h] = v;
        }
        __syncthreads();  // red_max reads done, p_s written
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < kGMax; ++h) red_sum[warp][h] = psum[h];
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < kGMax; ++h) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < kSimtThreads / 32; ++w) s += red_sum[w][h];
            l_run[h] = l_run[h] * alpha[h] + s;
            m_run[h] = mnew[h];
#pragma unroll
            for (int j = 0; j < DPT; ++j) acc[h][j] *= alpha[h];
        }
        // ---- P.V: this thread's head_dim elements, all heads
        const int nt = min(kSimtTile, t_end - t0);
#pragma unroll
        for (int j = 0; j < DPT; ++j) {
            const int d = tid + j * kSimtThreads;
            if (d < D) {
                const int g = d / kGroup;
                for (int k = 0; k < nt; ++k) {
                    const long long r = row0 + t0 + k;
                    const uint8_t byte = p.v_codes[r * (D / 2) + d / 2];
                    const float code = static_cast<float>((d & 1) ? (byte >> 4) : (byte & 0xf));
                    const float v = fmaf(__half2float(__ushort_as_half(p.v_scale[r * NG + g])), code,
                                         __half2float(__ushort_as_half(p.v_bias[r * NG + g])));
#pragma unroll
                    for (int h = 0; h < kGMax; ++h) acc[h][j] = fmaf(p_s[k][h], v, acc[h][j]);
                }
            }
        }
        __syncthreads();  // p_s / red_sum reused by the next tile
    }

    // ---- write this split's partial state (natural-log units for m)
    const float ln2 = 0.69314718055994531f;
#pragma unroll
    for (int h = 0; h < kGMax; ++h) {
        if (h >= G) continue;
        const long long ph = (static_cast<long long>(b) * p.num_q_heads + kvh * G + h) * p.n_splits + split;
#pragma unroll
        for (int j = 0; j < DPT; ++j) {
            const int d = tid + j * kSimtThreads;
            if (d < D) p.part_acc[ph * D + d] = acc[h][j];
        }
        if (tid == 0) {
            p.part_m[ph] = m_run[h] == -INFINITY ? -INFINITY : m_run[h] * ln2;
            p.part_l[ph] = l_run[h];
        }
    }
}

}  // namespace

int simt_ctas_per_sm(int head_dim) {
    int n = 0;
    switch (head_dim) {
        case 64: cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<64>, kSimtThreads, 0); break;
        case 128: cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<128>, kSimtThreads, 0); break;
        case 256: cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<256>, kSimtThreads, 0); break;
    }
    return n > 0 ? n : 1;
}

cudaError_t launch_decode_simt(const DecodeParams& p, int head_dim, cudaStream_t stream) {
    dim3 grid(p.n_splits, p.num_kv_heads, p.batch);
    switch (head_dim) {
        case 64: decode_simt_kernel<64><<<grid, kSimtThreads, 0, stream>>>(p); break;
        case 128: decode_simt_kernel<128><<<grid, kSimtThreads, 0, stream>>>(p); break;
        case 256: decode_simt_kernel<256><<<grid, kSimtThreads, 0, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace tq

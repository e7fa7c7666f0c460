// reduce.cu -- split-K phase 2: log-sum-exp merge of partial softmax states
// ("turboquant-llama3.170B" README, split-K paragraph: Phase 2 reduces the
// partial softmax results of the chunks processed in parallel by Phase 1).
//
// Per (b, h):  M = max_c m_c over parts with l_c > 0,  w_c = e^{m_c - M},
//              out = sum_c w_c acc_c / sum_c w_c l_c   (fp16, RNE; 0 if empty)
// One CTA per (b, h): reduce_fast_kernel for up to 64 parts (one round trip;
// barriers only for the output rotation's cross-warp stages), reduce_kernel
// beyond.
// Launched as a programmatic dependent of phase 1, each waits for phase 1's
// memory before the first read.
#include <math.h>

#include <atomic>

#include "tq_device.cuh"
#include "tq_hadamard.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kReduceThreads = 256;
constexpr int kReduceWarps = kReduceThreads / 32;

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kReduceWarps; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    __syncthreads();
    return r;
}

// Warp w sums parts w, w + 8, ...; lane owns head_dim elements
// [lane * V, lane * V + V), read with vector loads; the eight warp sums are
// combined through shared memory.  The first R rows of every warp are loaded
// before the weights are known, so the row reads overlap the max / sum
// reductions instead of following them.
template <int D>
__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(const ReduceParams p) {
    constexpr int V = D / 32;  // floats per lane per row
    constexpr int R = 48 / V;  // rows per warp in flight
    extern __shared__ float w_s[];  // [n_parts]: m, then the weight of each part
    __shared__ float red[kReduceWarps];
    __shared__ float part_sum[kReduceWarps][D];
    pdl_wait_primary();
    // phase 1 is complete: an eager next step's phase 1 may launch now (it
    // waits for this grid before its first read)
    pdl_launch_dependents();
    const long long bh = blockIdx.x;
    if (p.adv_n != 0 && threadIdx.x == 0 && bh % p.num_q_heads == 0) {  // phase 1 has read the lengths
        const long long b = bh / p.num_q_heads;
        p.adv_seq_lens[b] += p.adv_n;
        p.adv_write_pos[b] += p.adv_n;
    }
    const int n = p.n_parts;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float* pm = p.part_m + bh * n;
    const float* pl = p.part_l + bh * n;
    const float* pa = p.part_acc + bh * n * D;
    float x[R][V];
    auto load_rows = [&](int base) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int c = base + warp + r * kReduceWarps;
            if (c < n) {
                const float* src = pa + static_cast<long long>(c) * D + lane * V;
                if constexpr (V == 2) {
                    const float2 v = *reinterpret_cast<const float2*>(src);
                    x[r][0] = v.x; x[r][1] = v.y;
                } else {
#pragma unroll
                    for (int i = 0; i < V; i += 4) {
                        const float4 v = *reinterpret_cast<const float4*>(src + i);
                        x[r][i] = v.x; x[r][i + 1] = v.y; x[r][i + 2] = v.z; x[r][i + 3] = v.w;
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) x[r][i] = 0.0f;
            }
        }
    };
    load_rows(0);
    float M = -INFINITY;
    for (int c = threadIdx.x; c < n; c += kReduceThreads) {
        const float m = pl[c] > 0.0f ? pm[c] : -INFINITY;  // empty parts carry no weight
        w_s[c] = m;
        M = fmaxf(M, m);
    }
    M = block_reduce(M, red, true);
    float L = 0.0f;
    for (int c = threadIdx.x; c < n; c += kReduceThreads) {
        const float m = w_s[c];
        const float w = m == -INFINITY ? 0.0f : expf(m - M);
        w_s[c] = w;
        L = fmaf(w, pl[c], L);
    }
    L = block_reduce(L, red, false);  // its barriers also publish w_s
    float a[V];
#pragma unroll
    for (int i = 0; i < V; ++i) a[i] = 0.0f;
    for (int base = 0; base < n; base += R * kReduceWarps) {
        if (base > 0) load_rows(base);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int c = base + warp + r * kReduceWarps;
            const float w = c < n ? w_s[c] : 0.0f;
            if (w != 0.0f) {  // same branch for the whole warp
#pragma unroll
                for (int i = 0; i < V; ++i) a[i] = fmaf(w, x[r][i], a[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < V; ++i) part_sum[warp][lane * V + i] = a[i];
    __syncthreads();
    if (!p.rotate_out) {
        for (int d = threadIdx.x; d < D; d += kReduceThreads) {
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < kReduceWarps; ++w) t += part_sum[w][d];
            p.out[bh * D + d] = __half_as_ushort(__float2half_rn(L > 0.0f ? __fdiv_rn(t, L) : 0.0f));
        }
        return;
    }
    // values were stored rotated: the output is H applied to the merged fp32
    // output (warp 0, V consecutive elements per lane), rounded once to fp16
    if (warp == 0) {
        float o[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < kReduceWarps; ++w) t += part_sum[w][lane * V + i];
            o[i] = L > 0.0f ? __fdiv_rn(t, L) : 0.0f;
        }
        hadamard_warp<V>(o, lane, p.rot_scale);
#pragma unroll
        for (int i = 0; i < V; ++i) p.out[bh * D + lane * V + i] = __half_as_ushort(__float2half_rn(o[i]));
    }
}

// Up to 64 parts (19 at 128K in the one-CTA-per-SM layout, 43 at 16K in the
// three-CTA one): one thread per head_dim element loads its element of every
// part and each warp the parts' m and l at once, one round trip to L2, then
//   M = warp max over lanes (lane c holds parts c and c + 32),
//   w_c = expf(m_c - M),
//   L = xor-tree warp sum of fmaf(w_c, l_c, 0) + fmaf(w_c+32, l_c+32, 0),
//   t = sum over parts in order of fmaf(w_c, acc_c, 0) (w_c = 0 skipped),
// no CTA barrier (but for ROT below).  Up to 32 parts M, w and L are
// reduce_kernel's (its block reduction sees the same 32 values, the other
// warps' zeros added exactly), and t its too up to 8 parts (one part per warp
// there), so the two give the same bits up to 8 parts, as does the cluster
// merge in phase 1.  (reduce_kernel: 2.0-2.2 us after its release for 19 or
// 43 parts, five barriers and dependent loads.)
//   Its CTAs are launched while phase 1 runs and take SMs as phase-1 CTAs
// leave; small as they are, the first SMs to free up would take seven each,
// and their loads queue there (128K step 32.8 us, against 31.0 us spread).
// Each CTA therefore reserves kFastSmemPad bytes of shared memory it does not
// use, so that at most two share an SM (grids of up to two CTAs per SM; a
// batch's larger grid runs unpadded: ragged batch of 32, 110.7 -> 106.7 us).
//   ROT (values stored rotated): the output is H applied to the merged fp32
// output, then the scale and one fp16 rounding, with the stages in increasing
// order h = 1, 2, ..., D / 2 and each butterfly one round-to-nearest add or
// subtract, as in reduce_kernel: element d = thread + j * TH, so stages
// h < 32 pair lanes (shuffles), 32 <= h < TH pair warps (shared memory) and
// h = TH (head_dim 256) pairs a thread's two elements.  Given the same merged
// values both rotate to the same bits.
constexpr int kFastParts = 64;
constexpr int kFastSmemPad = 100 * 1024;

template <int D, bool ROT>
__global__ void __launch_bounds__(D < 128 ? D : 128) reduce_fast_kernel(const ReduceParams p) {
    constexpr int TH = D < 128 ? D : 128;
    constexpr int DPT = D / TH;  // head_dim elements per thread
    __shared__ float xs[ROT ? D : 1];  // ROT: one cross-warp stage's values
    pdl_wait_primary();
    // phase 1 is complete: an eager next step's phase 1 may launch now (it
    // waits for this grid before its first read)
    pdl_launch_dependents();
    const long long bh = blockIdx.x;
    if (p.adv_n != 0 && threadIdx.x == 0 && bh % p.num_q_heads == 0) {  // phase 1 has read the lengths
        const long long b = bh / p.num_q_heads;
        p.adv_seq_lens[b] += p.adv_n;
        p.adv_write_pos[b] += p.adv_n;
    }
    const int n = p.n_parts;
    const int lane = threadIdx.x & 31;
    const float* pa = p.part_acc + bh * n * D + threadIdx.x;
    float a[kFastParts][DPT];
#pragma unroll
    for (int c = 0; c < kFastParts; ++c) {
#pragma unroll
        for (int j = 0; j < DPT; ++j) a[c][j] = c < n ? __ldcg(pa + c * D + j * TH) : 0.0f;
    }
    float l[2], m[2], w[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int c = lane + 32 * i;
        l[i] = c < n ? __ldcg(p.part_l + bh * n + c) : 0.0f;
        const float mv = c < n ? __ldcg(p.part_m + bh * n + c) : -INFINITY;
        m[i] = l[i] > 0.0f ? mv : -INFINITY;  // empty parts carry no weight
    }
    float M = fmaxf(m[0], m[1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
#pragma unroll
    for (int i = 0; i < 2; ++i) w[i] = m[i] == -INFINITY ? 0.0f : expf(m[i] - M);
    float L = fmaf(w[0], l[0], 0.0f) + fmaf(w[1], l[1], 0.0f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    float t[DPT];
#pragma unroll
    for (int j = 0; j < DPT; ++j) t[j] = 0.0f;
#pragma unroll
    for (int c = 0; c < kFastParts; ++c) {
        const float wc = __shfl_sync(0xffffffffu, w[c / 32], c & 31);
        if (c < n && wc != 0.0f) {
#pragma unroll
            for (int j = 0; j < DPT; ++j) t[j] += fmaf(wc, a[c][j], 0.0f);
        }
    }
    float o[DPT];
#pragma unroll
    for (int j = 0; j < DPT; ++j) o[j] = L > 0.0f ? __fdiv_rn(t[j], L) : 0.0f;
    if constexpr (ROT) {
        const int x = threadIdx.x;
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {  // the partner element in lane ^ h
#pragma unroll
            for (int j = 0; j < DPT; ++j) {
                const float other = __shfl_xor_sync(0xffffffffu, o[j], h);
                o[j] = (x & h) != 0 ? __fsub_rn(other, o[j]) : __fadd_rn(o[j], other);
            }
        }
#pragma unroll
        for (int h = 32; h < TH; h <<= 1) {  // the partner element in another warp
#pragma unroll
            for (int j = 0; j < DPT; ++j) xs[x + j * TH] = o[j];
            __syncthreads();
#pragma unroll
            for (int j = 0; j < DPT; ++j) {
                const float other = xs[(x ^ h) + j * TH];
                o[j] = (x & h) != 0 ? __fsub_rn(other, o[j]) : __fadd_rn(o[j], other);
            }
            __syncthreads();
        }
        if constexpr (DPT == 2) {  // h = TH: this thread's elements x and x + TH
            const float u = o[0], w = o[1];
            o[0] = __fadd_rn(u, w);
            o[1] = __fsub_rn(u, w);
        }
#pragma unroll
        for (int j = 0; j < DPT; ++j) o[j] = __fmul_rn(o[j], p.rot_scale);
    }
#pragma unroll
    for (int j = 0; j < DPT; ++j) p.out[bh * D + threadIdx.x + j * TH] = __half_as_ushort(__float2half_rn(o[j]));
}

// TQ_STEP_ADVANCE after a step whose append ran as its own kernel: a plain
// launch after the reduce, so stream order covers the append as well.
__global__ void advance_lengths_kernel(int32_t* seq_lens, int32_t* write_pos, int batch, int n) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) {
        seq_lens[b] += n;
        write_pos[b] += n;
    }
}

}  // namespace

cudaError_t launch_advance(int32_t* seq_lens, int32_t* write_pos, int batch, int n, cudaStream_t stream) {
    advance_lengths_kernel<<<(batch + 127) / 128, 128, 0, stream>>>(seq_lens, write_pos, batch, n);
    return cudaGetLastError();
}

// The fast reduce's shared-memory reservation, once per device.
cudaError_t fast_attrs() {
    static std::atomic<bool> done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    const bool cache = dev >= 0 && dev < 64;
    if (cache && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    using Kern = void (*)(ReduceParams);
    const Kern kerns[6] = {reduce_fast_kernel<64, false>,  reduce_fast_kernel<128, false>,
                           reduce_fast_kernel<256, false>, reduce_fast_kernel<64, true>,
                           reduce_fast_kernel<128, true>,  reduce_fast_kernel<256, true>};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 6 && e == cudaSuccess; ++i)
        e = cudaFuncSetAttribute(kerns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, kFastSmemPad);
    if (e == cudaSuccess && cache) done[dev].store(true, std::memory_order_release);
    return e;
}

cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream, bool pdl_secondary) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.num_q_heads);
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(p.n_parts) * sizeof(float);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_secondary ? 1 : 0;
    if (p.n_parts <= kFastParts) {
        cfg.blockDim = dim3(p.head_dim < 128 ? p.head_dim : 128);
        // the spreading pad only while the grid fits in two CTAs per SM: a
        // larger grid (a batch) runs in waves anyway, and padded CTAs would
        // only make more of them
        static std::atomic<int> sm_n[64];
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        if (dev >= 0 && dev < 64) sms = sm_n[dev].load(std::memory_order_relaxed);
        if (sms == 0) {
            const cudaError_t ea = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (ea != cudaSuccess) return ea;
            if (dev >= 0 && dev < 64) sm_n[dev].store(sms, std::memory_order_relaxed);
        }
        cfg.dynamicSmemBytes = cfg.gridDim.x <= 2u * static_cast<unsigned>(sms) ? kFastSmemPad : 0;
        const cudaError_t e = fast_attrs();
        if (e != cudaSuccess) return e;
        using Kern = void (*)(ReduceParams);
        Kern k = nullptr;
        const bool rot = p.rotate_out != 0;
        switch (p.head_dim) {
            case 64: k = rot ? reduce_fast_kernel<64, true> : reduce_fast_kernel<64, false>; break;
            case 128: k = rot ? reduce_fast_kernel<128, true> : reduce_fast_kernel<128, false>; break;
            case 256: k = rot ? reduce_fast_kernel<256, true> : reduce_fast_kernel<256, false>; break;
            default: return cudaErrorInvalidValue;
        }
        return cudaLaunchKernelEx(&cfg, k, p);
    }
    switch (p.head_dim) {
        case 64: return cudaLaunchKernelEx(&cfg, reduce_kernel<64>, p);
        case 128: return cudaLaunchKernelEx(&cfg, reduce_kernel<128>, p);
        case 256: return cudaLaunchKernelEx(&cfg, reduce_kernel<256>, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tq

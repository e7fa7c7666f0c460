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
#include <atomic>

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

// Destination of group gi (over [B][Hkv][n_new][NG]) in the cache: the code
// and scale / bias offsets of its row write_pos[b] + i; false (and the status
// bit) when the sequence's write position is out of range.
template <int BITS>
__device__ __forceinline__ bool group_dst(const AppendParams& p, long long gi, int ng, long long& code_off,
                                          long long& sb) {
    const long long row = fast_div(gi, p.div_ng);  // over [B][Hkv][n_new]
    const int g = static_cast<int>(gi - row * ng);
    const long long bh = fast_div(row, p.div_n_new);  // b * Hkv + h
    const int i = static_cast<int>(row - bh * p.n_new);
    const int b = static_cast<int>(fast_div(bh, p.div_hkv));
    const int wp = __ldg(p.write_pos + b);
    if (wp < 0 || static_cast<long long>(wp) + p.n_new > p.capacity) {
        if (p.status != nullptr && g == 0 && i == 0) atomicOr(p.status, TQ_DEV_WRITE_POS);
        return false;
    }
    const long long dst_row =
        kv_row(p.map, p.num_kv_heads, b, static_cast<int>(bh - static_cast<long long>(b) * p.num_kv_heads), wp + i,
               p.status);
    code_off = dst_row * (p.head_dim * BITS / 8) + g * (kGroup * BITS / 8);  // 32-byte aligned
    sb = dst_row * ng + g;
    return true;
}

// Quantize one group's 64 fp16 values (eight 16-byte words) of tensor t (0: K,
// 1: V) and store codes, scale and bias.
template <int BITS>
__device__ __forceinline__ void quantize_words_store(const AppendParams& p, const uint4 (&x)[8], int t,
                                                     long long code_off, long long sb) {
    uint32_t c[2 * BITS];
    __half sc, bi;
    quantize_group64<BITS>(x, c, sc, bi);
    uint4* dst = reinterpret_cast<uint4*>((t ? p.v_codes : p.k_codes) + code_off);
#pragma unroll
    for (int w = 0; w < BITS / 2; ++w) dst[w] = make_uint4(c[4 * w], c[4 * w + 1], c[4 * w + 2], c[4 * w + 3]);
    (t ? p.v_scale : p.k_scale)[sb] = __half_as_ushort(sc);
    (t ? p.v_bias : p.k_bias)[sb] = __half_as_ushort(bi);
}

// Quantize group gi from its staged K and V rows (eight 16-byte words each,
// word j at slot j ^ r7) and store it into the cache row write_pos[b] + i.
template <int BITS>
__device__ __forceinline__ void quantize_store(const AppendParams& p, long long gi, int ng, const uint4* rowk,
                                               const uint4* rowv, int r7, int t_first = 0, int t_last = 1) {
    long long code_off, sb;
    if (!group_dst<BITS>(p, gi, ng, code_off, sb)) return;
#pragma unroll 1
    for (int t = t_first; t <= t_last; ++t) {  // 0: K, 1: V
        const uint4* src = t ? rowv : rowk;
        uint4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = src[j ^ r7];
        quantize_words_store<BITS>(p, x, t, code_off, sb);
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
    quantize_store<BITS>(p, gi, ng, stage[warp][0][lane], stage[warp][1][lane], lane & 7);
}

// The Hadamard rotation of a row whose NG groups of 64 are held by NG
// consecutive lanes, this thread holding group g in v (fp32).  The stages run
// in the order of the fast transform (h = 1, 2, ..., 32 inside the thread,
// then h = 64, 128 with the lanes lane ^ 1, lane ^ 2), each butterfly one
// round-to-nearest add and one subtract (two butterflies per paired fp32
// operation), so the result equals the sequential transform bit for bit; then
// the scale.  Every lane of the warp takes part.
template <int NG>
__device__ __forceinline__ void rotate_group_thread(float (&v)[64], int g, float scale) {
    const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int i = 0; i < 64; i += 4) {  // h = 1: butterflies (i, i+1) and (i+2, i+3) in one paired op each
        const float2 a = make_float2(v[i], v[i + 2]), b = make_float2(v[i + 1], v[i + 3]);
        const float2 sum = __fadd2_rn(a, b), dif = __ffma2_rn(b, m1, a);
        v[i] = sum.x;
        v[i + 2] = sum.y;
        v[i + 1] = dif.x;
        v[i + 3] = dif.y;
    }
#pragma unroll
    for (int h = 2; h < 64; h <<= 1) {  // pairs (i, i+1) with bit h clear: two butterflies per paired op
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
            if ((i & h) != 0) continue;
            const float2 a = make_float2(v[i], v[i + 1]), b = make_float2(v[i + h], v[i + h + 1]);
            const float2 sum = __fadd2_rn(a, b), dif = __ffma2_rn(b, m1, a);
            v[i] = sum.x;
            v[i + 1] = sum.y;
            v[i + h] = dif.x;
            v[i + h + 1] = dif.y;
        }
    }
#pragma unroll
    for (int hl = 1; hl < NG; hl <<= 1) {  // h = 64 * hl: the group in lane ^ hl
        // lower lane: v + other; upper lane: other - v; both one rounding of
        // fma(v, c, other) with c = +1 / -1 (exact products)
        const float c = (g & hl) != 0 ? -1.0f : 1.0f;
        const float2 c2 = make_float2(c, c);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
            const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, v[i], hl),
                                         __shfl_xor_sync(0xffffffffu, v[i + 1], hl));
            const float2 r = __ffma2_rn(make_float2(v[i], v[i + 1]), c2, o);
            v[i] = r.x;
            v[i + 1] = r.y;
        }
    }
    const float2 sc = make_float2(scale, scale);
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
        const float2 r = __fmul2_rn(make_float2(v[i], v[i + 1]), sc);
        v[i] = r.x;
        v[i + 1] = r.y;
    }
}

// Rotate a staged group (slots j ^ r7) in registers and quantize it.
template <int BITS, int NG>
__device__ __forceinline__ void rotate_quantize_store(const AppendParams& p, long long gi, int g, const uint4* row,
                                                      int r7, int t) {
    float v[64];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 w = row[j ^ r7];
        const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(h[k]);
            v[8 * j + 2 * k] = f.x;
            v[8 * j + 2 * k + 1] = f.y;
        }
    }
    rotate_group_thread<NG>(v, g, p.rot_scale);  // all lanes, before any exit
    uint4 x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __half2 h = __floats2half2_rn(v[8 * j + 2 * k], v[8 * j + 2 * k + 1]);
            w[k] = *reinterpret_cast<const uint32_t*>(&h);
        }
        x[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    long long code_off, sb;
    if (gi >= 0 && group_dst<BITS>(p, gi, NG, code_off, sb)) quantize_words_store<BITS>(p, x, t, code_off, sb);
}

// Large appends (prefill): a persistent grid streams tiles of kTmaGroups
// groups of K and of V into shared memory with 2-D TMA boxes (128-byte rows,
// one group per row).  The 128-byte swizzle places word j of row r at slot
// j ^ (r & 7), the layout the per-thread reads above expect.  Two stages per
// CTA: while the threads quantize one tile, the next one is in flight.  A
// stage is released warp by warp (a shared count, no CTA barrier): the last
// warp to finish with it issues its refill, and the other warps go on to the
// next stage meanwhile.
constexpr int kTmaGroups = 128;                     // groups (rows) per tile
constexpr int kTmaThreads = 2 * kTmaGroups;         // one thread per (group, K or V)
constexpr int kTmaTensorBytes = kTmaGroups * 128;   // 16 KB of K or of V
constexpr int kTmaStageBytes = 2 * kTmaTensorBytes;
constexpr int kTmaStages = 2;
constexpr int kTmaSmemBytes = kTmaStages * kTmaStageBytes + 1024;
constexpr int kTmaWarps = kTmaThreads / 32;

template <int BITS, bool ROT>
__global__ void __launch_bounds__(kTmaThreads, ROT ? 2 : 3) quantize_append_tma_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                         const __grid_constant__ CUtensorMap tm_v,
                                                                         const AppendParams p, long long n_groups,
                                                                         int n_tiles) {
    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[kTmaStages];
    __shared__ unsigned int done_cnt[kTmaStages];  // warps finished with the stage, cumulative
    uint8_t* smem = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
    const int tid = threadIdx.x, lane = tid & 31;
    const int ng = p.head_dim / kGroup;
    if (tid == 0) {
        for (int s = 0; s < kTmaStages; ++s) {
            mbar_init(&full_bar[s], 1);
            done_cnt[s] = 0;
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    auto issue = [&](int tile, int stage) {
        const uint64_t policy = policy_evict_first();
        uint8_t* st = smem + stage * kTmaStageBytes;
        mbar_arrive_expect_tx(&full_bar[stage], kTmaStageBytes);
        tma_load_2d(st, &tm_k, 0, tile * kTmaGroups, &full_bar[stage], policy);
        tma_load_2d(st + kTmaTensorBytes, &tm_v, 0, tile * kTmaGroups, &full_bar[stage], policy);
    };
    if (tid == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        for (int s = 0; s < kTmaStages; ++s)
            if (blockIdx.x + s * gridDim.x < n_tiles) issue(blockIdx.x + s * gridDim.x, s);
    }
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
        const int stage = it % kTmaStages;
        if (!mbar_wait_bounded(&full_bar[stage], (it / kTmaStages) & 1)) {
            if (p.status != nullptr) atomicOr(p.status, TQ_DEV_TIMEOUT);
            break;  // no further tiles are issued, so every thread gives up the same way
        }
        uint4 (*tk)[8] = reinterpret_cast<uint4 (*)[8]>(smem + stage * kTmaStageBytes);
        uint4 (*tv)[8] = reinterpret_cast<uint4 (*)[8]>(smem + stage * kTmaStageBytes + kTmaTensorBytes);
        // threads [0, 128) take the K groups, [128, 256) the V groups
        const int t = tid >= kTmaGroups ? 1 : 0, r = tid - t * kTmaGroups;
        const long long gi = static_cast<long long>(tile) * kTmaGroups + r;
        if (ROT && (p.flags & (t ? TQ_ROTATE_V : TQ_ROTATE_K))) {  // the same for each warp
            // every lane rotates (the shuffles need the whole warp); lanes past
            // the last group hold zero-filled rows and store nothing
            const long long gq = gi < n_groups ? gi : -1;
            switch (ng) {
                case 1: rotate_quantize_store<BITS, 1>(p, gq, r % 1, (t ? tv : tk)[r], r & 7, t); break;
                case 2: rotate_quantize_store<BITS, 2>(p, gq, r % 2, (t ? tv : tk)[r], r & 7, t); break;
                default: rotate_quantize_store<BITS, 4>(p, gq, r % 4, (t ? tv : tk)[r], r & 7, t); break;
            }
        } else if (gi < n_groups) {
            quantize_store<BITS>(p, gi, ng, tk[r], tv[r], r & 7, t, t);
        }
        // Release the stage (this thread only read it).  The last warp to
        // finish it refills it: its fences order every warp's reads (made
        // visible by their fences before the count) before the asynchronous
        // copy that overwrites the stage.
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const unsigned int before = atomicAdd(&done_cnt[stage], 1u);
            const int next = tile + kTmaStages * gridDim.x;
            if (before % kTmaWarps == kTmaWarps - 1 && next < n_tiles) {
                __threadfence_block();
                fence_proxy_async_shared();
                issue(next, stage);
            }
        }
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

cudaError_t launch_quantize_append_tma(const AppendParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                       int grid, cudaStream_t stream) {
    const long long groups = static_cast<long long>(p.batch) * p.num_kv_heads * p.n_new * (p.head_dim / kGroup);
    const long long tiles = (groups + kTmaGroups - 1) / kTmaGroups;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int n_tiles = static_cast<int>(tiles);
    if (grid > n_tiles) grid = n_tiles;
    if (grid < 1) return cudaSuccess;
    const bool rot = (p.flags & (TQ_ROTATE_K | TQ_ROTATE_V)) != 0;
    if (rot) grid = grid * 2 / 3;  // the rotating instantiation runs 2 CTAs per SM (registers)
    if (grid < 1) grid = 1;
    static std::atomic<bool> attr_done[64][4];  // per device and variant; a repeated set is harmless
    int dev = 0;
    cudaGetDevice(&dev);
    const int vi = (p.bits == 8 ? 1 : 0) + (rot ? 2 : 0);
    auto kern = [&]() {
        if (p.bits == 8) return rot ? quantize_append_tma_kernel<8, true> : quantize_append_tma_kernel<8, false>;
        return rot ? quantize_append_tma_kernel<4, true> : quantize_append_tma_kernel<4, false>;
    }();
    if (dev >= 0 && dev < 64 && !attr_done[dev][vi].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTmaSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev][vi].store(true, std::memory_order_release);
    }
    kern<<<grid, kTmaThreads, kTmaSmemBytes, stream>>>(tm_k, tm_v, p, groups, n_tiles);
    return cudaGetLastError();
}

cudaError_t launch_quantize_append_primary(const AppendParams& p, cudaStream_t stream) {
    return launch_quantize_append(p, stream);
}

}  // namespace tq

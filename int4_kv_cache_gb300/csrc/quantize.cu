// quantize.cu -- quantize-on-store: fp16 K/V rows -> packed int4 codes plus
// fp16 scale/bias per group of 64, written in place into the cache.
//
// Method: "turboquant-llama3.170B" README, decode-step listing (quantize K,V to
// int4 after RoPE, then store) and the Gemma page, Background (MLX-style int4
// with a per-group scale and bias).  The rounding rule is the one stated in
// tq.h; every step is a single IEEE fp32 operation with round-to-nearest-even,
// so codes, scales and biases are bit-identical to the CPU oracle.  The
// per-element division is replaced by two fused multiply-adds with multipliers
// bracketing 1/scale wherever they provably give the division's code
// (tq_quant.cuh).
//
// Work split: one thread per (row, group of 64): it takes the group of K and
// the group of V (eight 16-byte words each) and writes 32 bytes of codes per
// tensor and the four scale / bias halves.  With no cross-lane reductions the
// per-group work (min/max, the scale division, the reciprocal) is spread over
// 64 elements.  Small appends stage each warp's groups through shared memory
// with coalesced loads; prefills stream 256-row tiles by TMA (below).
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
                                               const uint4* rowv, int r7) {
    long long code_off, sb;
    if (!group_dst<BITS>(p, gi, ng, code_off, sb)) return;
#pragma unroll 1
    for (int t = 0; t < 2; ++t) {  // 0: K, 1: V
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

// Large appends (prefill): a persistent grid streams tiles of ROWS rows of
// 128 bytes (one group of 64 fp16 values per row) of K and of V into shared
// memory with 2-D TMA boxes.  The 128-byte swizzle places word j of row r at
// slot j ^ (r & 7).  One thread per row takes the group of K, then the group
// of V (both go to the same cache offsets, found once).  K and V have a
// buffer each: a thread copies its group into registers and releases the
// buffer at once; the last warp to release it issues the next tile's copy
// into it, which then lands while the CTA works on the other tensor.  The
// release is counted per warp (no CTA barrier).
template <int ROWS, int WARPS>
struct KVTiles {
    static constexpr int kTensorBytes = ROWS * 128;
    static constexpr int kSmemBytes = 2 * kTensorBytes + 1024;

    uint8_t* smem;  // 1024-byte aligned (the swizzle pattern repeats every 1024 bytes)
    uint64_t* full_bar;      // [2]: K, V
    unsigned int* done_cnt;  // [2]: warps finished with the buffer, cumulative
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    int n_tiles;

    __device__ __forceinline__ void issue(int tile, int t) const {
        mbar_arrive_expect_tx(&full_bar[t], kTensorBytes);
        tma_load_2d(smem + t * kTensorBytes, t ? tm_v : tm_k, 0, tile * ROWS, &full_bar[t], policy_evict_first());
    }
    // Barriers, then the first tile in flight; every thread of the CTA calls it.
    __device__ __forceinline__ void start() const {
        if (threadIdx.x == 0) {
            for (int t = 0; t < 2; ++t) {
                mbar_init(&full_bar[t], 1);
                done_cnt[t] = 0;
            }
            fence_mbarrier_init();
        }
        __syncthreads();
        pdl_launch_dependents();
        if (threadIdx.x == 0 && blockIdx.x < n_tiles) {
            prefetch_tensormap(tm_k);
            prefetch_tensormap(tm_v);
            issue(blockIdx.x, 0);
            issue(blockIdx.x, 1);
        }
    }
    // Tensor t of this CTA's it-th tile has landed (false: the bounded wait gave up).
    __device__ __forceinline__ bool wait(int it, int t) const { return mbar_wait_bounded(&full_bar[t], it & 1); }
    __device__ __forceinline__ const uint4 (*rows(int t) const)[8] {
        return reinterpret_cast<const uint4(*)[8]>(smem + t * kTensorBytes);
    }
    // This warp is done reading buffer t.  The last warp to finish it refills
    // it: its fences order every warp's reads (made visible by their fences
    // before the count) before the asynchronous copy that overwrites it.
    __device__ __forceinline__ void release(int tile, int t) const {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
            __threadfence_block();
            const unsigned int before = atomicAdd(&done_cnt[t], 1u);
            const int next = tile + gridDim.x;
            if (before % WARPS == WARPS - 1 && next < n_tiles) {
                __threadfence_block();
                fence_proxy_async_shared();
                issue(next, t);
            }
        }
    }
};

constexpr int kTmaGroups = kTmaAppendBoxRows;  // rows per tile
constexpr int kTmaThreads = kTmaGroups;        // one thread per row: its K group, then its V group
constexpr int kTmaWarps = kTmaThreads / 32;
using AppendTiles = KVTiles<kTmaGroups, kTmaWarps>;

template <int ROWS, int WARPS>
__device__ __forceinline__ KVTiles<ROWS, WARPS> kv_tiles(uint8_t* dyn_smem, uint64_t* full_bar, unsigned int* done_cnt,
                                                        const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                                        int n_tiles) {
    KVTiles<ROWS, WARPS> r;
    r.smem = dyn_smem + ((1024u - (smem_u32(dyn_smem) & 1023u)) & 1023u);
    r.full_bar = full_bar;
    r.done_cnt = done_cnt;
    r.tm_k = tm_k;
    r.tm_v = tm_v;
    r.n_tiles = n_tiles;
    return r;
}

template <int BITS>
__global__ void __launch_bounds__(kTmaThreads, 3)
    quantize_append_tma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                               const AppendParams p, long long n_groups, int n_tiles) {
    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[2];
    __shared__ unsigned int done_cnt[2];
    const AppendTiles tiles = kv_tiles<kTmaGroups, kTmaWarps>(dyn_smem, full_bar, done_cnt, &tm_k, &tm_v, n_tiles);
    tiles.start();
    const int ng = p.head_dim / kGroup, r = threadIdx.x;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
        const long long gi = static_cast<long long>(tile) * kTmaGroups + r;
        long long code_off = 0, sb = 0;
        const bool ok = gi < n_groups && group_dst<BITS>(p, gi, ng, code_off, sb);
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
            if (!tiles.wait(it, t)) {
                if (p.status != nullptr) atomicOr(p.status, TQ_DEV_TIMEOUT);
                return;  // no further tiles are issued, so every thread gives up the same way
            }
            uint4 x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = tiles.rows(t)[r][j ^ (r & 7)];
            tiles.release(tile, t);  // the group is in registers
            if (ok) quantize_words_store<BITS>(p, x, t, code_off, sb);
        }
    }
}

// ------------------------------------------------------------------------
// Rotated: the same one thread per group row (its K group, then its V group);
// a head row's NG groups sit in NG consecutive lanes ("Running and Evaluating
// TurboQuant optimized Gemma 4", TurboQuant section: x -> H x / sqrt(D) before
// quantisation).  The
// fast transform runs its stages in increasing order h = 1, 2, ..., D / 2,
// each butterfly one round-to-nearest fp32 add or subtract, then the scale
// and the fp16 rounding: the same operations as the sequential transform, so
// the stored rows are bit-identical to it.  Stages h < 64 run in the thread,
// h = 64, 128 between the lanes lane and lane ^ 1, lane ^ 2.
constexpr int kRotCtasPerSm = 2;  // registers: 64 fp32 values per thread

// x: the group's 64 fp16 values (eight 16-byte words) -> v: H x / sqrt(D) of
// this group's part of the row, fp32.
template <int NG>
__device__ __forceinline__ void rotate_group_thread(const uint4 (&x)[8], float (&v)[64], int g, float scale) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // h = 1 straight from fp16: x0 + x1, x0 - x1 with x1 widened once
        const __half2* hp = reinterpret_cast<const __half2*>(&x[j]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float u = __high2float(hp[e]);
            v[8 * j + 2 * e] = add_h_f(__low2half(hp[e]), u);
            v[8 * j + 2 * e + 1] = sub_h_f(__low2half(hp[e]), u);
        }
    }
    const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int h = 2; h < 64; h <<= 1) {  // pairs (i, i + 1) with bit h clear: two butterflies per paired op
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

template <int BITS, int NG>
__global__ void __launch_bounds__(kTmaThreads, kRotCtasPerSm)
    quantize_append_rot_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                               const AppendParams p, long long n_groups, int n_tiles) {
    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[2];
    __shared__ unsigned int done_cnt[2];
    const AppendTiles tiles = kv_tiles<kTmaGroups, kTmaWarps>(dyn_smem, full_bar, done_cnt, &tm_k, &tm_v, n_tiles);
    tiles.start();
    const int r = threadIdx.x;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
        const long long gi = static_cast<long long>(tile) * kTmaGroups + r;
        long long code_off = 0, sb = 0;
        const bool ok = gi < n_groups && group_dst<BITS>(p, gi, NG, code_off, sb);
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
            if (!tiles.wait(it, t)) {
                if (p.status != nullptr) atomicOr(p.status, TQ_DEV_TIMEOUT);
                return;  // no further tiles are issued, so every thread gives up the same way
            }
            uint4 x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = tiles.rows(t)[r][j ^ (r & 7)];
            tiles.release(tile, t);  // the group is in registers
            if ((p.flags & (t ? TQ_ROTATE_V : TQ_ROTATE_K)) != 0) {  // the same for the CTA
                // every lane (shuffles); lanes past the last group hold zero-filled rows
                float v[64];
                rotate_group_thread<NG>(x, v, r % NG, p.rot_scale);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    floats_to_halves<8>(*reinterpret_cast<const float(*)[8]>(&v[8 * j]), &x[j]);
            }
            if (ok) quantize_words_store<BITS>(p, x, t, code_off, sb);
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
                                       int sms, cudaStream_t stream) {
    const long long groups = static_cast<long long>(p.batch) * p.num_kv_heads * p.n_new * (p.head_dim / kGroup);
    const bool rot = (p.flags & (TQ_ROTATE_K | TQ_ROTATE_V)) != 0;
    const long long tiles = (groups + kTmaGroups - 1) / kTmaGroups;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int n_tiles = static_cast<int>(tiles);
    int grid = sms * (rot ? kRotCtasPerSm : kTmaAppendCtasPerSm);
    if (grid > n_tiles) grid = n_tiles;
    if (grid < 1) return cudaSuccess;
    using Kern = void (*)(CUtensorMap, CUtensorMap, AppendParams, long long, int);
    Kern kern = nullptr;
    int vi = 0;  // variant: code width x (plain, rotated head_dim 64 / 128 / 256)
    if (!rot) {
        kern = p.bits == 8 ? quantize_append_tma_kernel<8> : quantize_append_tma_kernel<4>;
        vi = 0;
    } else if (p.head_dim == 64) {
        kern = p.bits == 8 ? quantize_append_rot_kernel<8, 1> : quantize_append_rot_kernel<4, 1>;
        vi = 1;
    } else if (p.head_dim == 128) {
        kern = p.bits == 8 ? quantize_append_rot_kernel<8, 2> : quantize_append_rot_kernel<4, 2>;
        vi = 2;
    } else {
        kern = p.bits == 8 ? quantize_append_rot_kernel<8, 4> : quantize_append_rot_kernel<4, 4>;
        vi = 3;
    }
    vi = 2 * vi + (p.bits == 8 ? 1 : 0);
    const int smem = AppendTiles::kSmemBytes;
    static std::atomic<bool> attr_done[64][8];  // per device and variant; a repeated set is harmless
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev][vi].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_done[dev][vi].store(true, std::memory_order_release);
    }
    kern<<<grid, kTmaThreads, smem, stream>>>(tm_k, tm_v, p, groups, n_tiles);
    return cudaGetLastError();
}

cudaError_t launch_quantize_append_primary(const AppendParams& p, cudaStream_t stream) {
    return launch_quantize_append(p, stream);
}

}  // namespace tq

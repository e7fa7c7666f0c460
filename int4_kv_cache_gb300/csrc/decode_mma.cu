// decode_mma.cu -- split-K phase 1 of int4 decode attention on tensor cores.
//
// What it computes ("turboquant-llama3.170B" README, kernel + split-K
// paragraphs; "Fused int4 Attention for Gemma 4 31B", What I Built Instead):
// for one sequence b, one kv head and a run of whole chunks, the partial
// softmax state of every query head of the GQA group,
//     m = max_t s_t,  l = sum_t e^{s_t - m},  acc = sum_t e^{s_t - m} v_t,
// with s_t = attn_scale * q . k_t and k_t, v_t the dequantised cache rows
// (scale * code + bias per group of 64).  Dequantisation happens only in
// registers; no float K/V and no score matrix is written anywhere.
//
// GB300 design (not the Metal kernel's):
//  * Each tile (T tokens) of K codes, V codes and the four fp16 scale/bias
//    arrays streams into a ring of shared-memory stages: the code tiles by
//    2-D TMA with the 128-byte swizzle, the scale/bias rows by 1-D bulk
//    copies, completion on mbarriers.  There is no producer warp: the last
//    warp to finish a stage issues its refill, so every warp computes (one
//    CTA of twelve warps per SM for contiguous int4 caches at head_dim 128,
//    else several CTAs of four warps).  Every byte of the cache is read from
//    HBM once per step, with an evict-first L2 policy.
//  * Consumer warps turn the nibbles into fp16 operands with one AND per
//    register: a 4-bit code n in the low mantissa bits of a zero-exponent fp16
//    is the subnormal n * 2^-24, and the high nibble of a byte gives
//    16 n * 2^-24, so no integer->float conversion instruction is needed.
//  * The grouped scores use mma.sync m16n8k16 with M = 16 tokens, N = the 8
//    query heads of the GQA group (all heads share one read of K), K = 16
//    head_dim elements; each 64-element group accumulates separately so its
//    scale and bias are applied afterwards in fp32:
//        s_t = attn * sum_g (scale_tg * sum_{d in g} q_d n_td + bias_tg * sum_{d in g} q_d).
//    The high-nibble elements meet q/16 in the B operand (the pages' qdot
//    "pre-divide the query" idea), so all products carry the same 2^-24.
//  * P.V uses mma.sync with M = 16 head_dim elements, N = 8 heads, K = 16
//    tokens.  B = fp16(p_t * vscale_tg), built from the score fragments with
//    movmatrix (no shared-memory round trip); the bias part
//    sum_t p_t * vbias_tg, and the mean-code share of the fp16 rounding
//    error of B, are accumulated in fp32 on the side.  Each stage's code sum
//    is formed in fresh tensor-core accumulators and added to the running
//    state with round-to-nearest fp32 adds.
//  * Token order inside a 16-token tile and the head_dim order inside each
//    operand are chosen so that every ldmatrix is bank-conflict free against
//    the swizzled tile; the permutation is undone when the state is written.
#include <math.h>

#include <atomic>
#include <type_traits>

#include "tq_device.cuh"
#include "tq_hadamard.cuh"
#include "tq_internal.h"
#include "tq_quant.cuh"

namespace tq {

namespace {

constexpr uint32_t kLoNib = 0x000F000Fu;  // nibbles at bits 0..3 / 16..19 -> n * 2^-24
constexpr uint32_t kHiNib = 0x00F000F0u;  // nibbles at bits 4..7 / 20..23 -> 16 n * 2^-24
constexpr float kLazyMax = 8.0f;          // slack of the running softmax max (log2 units)
constexpr uint32_t kByte = 0x00FF00FFu;   // int8: bytes 0 and 2 of a register -> n * 2^-24

// The SM layouts of phase 1.  WIDE: one CTA of 12 warps per SM sharing one
// ring of 384-token stages, for contiguous int4 caches at head_dim 128 when
// the plan's grid is one wave over (nearly) every SM.  Three independent
// 4-warp CTAs on an SM finish at staggered times (the scheduler favours the
// first placed) and the SM runs its last stretch on one CTA; twelve warps
// releasing the same stages stay within a stage of each other, and a
// (sequence, kv head) needs a third as many runs.  At 128K: 152 CTAs of
// 6,912 tokens instead of 456 of 2,304, the step 33.4 -> 31.9 us; 2 CTAs of 6
// warps per SM measured 33.4 us, one of 8 warps with 6 stages 34.7 us.  In a
// grid of several waves an SM idles while its next CTA fills its ring, which
// three CTAs per SM hide (ragged batch of 32: 123 us wide against 109 us), and
// paged caches keep 128-token tiles (their pages hold whole tiles).
__host__ __device__ constexpr bool wide_ok(int D, int BITS, bool PAGED) { return D == 128 && BITS == 4 && !PAGED; }

template <int D, int BITS = 4, bool WIDE = false>
struct Cfg {
    static constexpr int NG = D / kGroup;          // scale/bias groups per row
    static constexpr int BPT = D * BITS / 8;       // code bytes per token
    static constexpr int SPT = BPT / 16;           // 16-byte segments per token
    static constexpr int EPS = 128 / BITS;         // elements per 16-byte segment
    // A code tile is HALVES column blocks of T rows of ROWB bytes, each laid
    // out by one TMA box with the 128-byte swizzle: one block (and TPR tokens
    // per 128-byte row) when a token's codes fit 128 bytes, two 128-byte
    // blocks for the 256-byte rows of int8 at head_dim 256.
    static constexpr int ROWB = BPT < 128 ? BPT : 128;
    static constexpr int HALVES = BPT / ROWB;
    static constexpr int SPR = ROWB / 16;          // 16-byte segments of a token in one block
    static constexpr int TPR = 128 / ROWB;         // tokens per 128-byte swizzle row (1 for 128-byte blocks)
    static constexpr int NWC = WIDE ? 12 : 4;      // warps (all consume; the last to finish a stage refills it)
    static constexpr int MT = (BPT >= 128) ? 1 : 2;  // 16-token m-tiles per warp per stage
    static constexpr float CODE_MEAN = ((1 << BITS) - 1) * 0.5f;  // mean of a code uniform on 0..L
    static constexpr int T = NWC * MT * 16;        // tokens per stage
    // 3 stages of 34 KB for the int8 head_dim-256 tiles keep 2 CTAs per SM; the
    // wide layout's ring of 3 stages of 54 KB measured 0.1-0.25 us faster per
    // decode than 4 (a shorter drain after the last tile lands), 2 slower at 128K
    static constexpr int STAGES = HALVES > 1 ? 3 : (WIDE ? 3 : 4);
    static constexpr int CODE_BYTES = T * BPT;     // one code tile (K or V)
    static constexpr int HALF_BYTES = T * ROWB;    // one column block of a code tile
    static constexpr int SB_BYTES = T * NG * 2;    // one scale or bias tile
    static constexpr int STAGE_BYTES = ((2 * CODE_BYTES + 4 * SB_BYTES + 1023) / 1024) * 1024;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;  // +1024 for base alignment
    static constexpr int THREADS = NWC * 32;
    static constexpr int NKS = D / 16;             // k-steps of the score MMA = m-tiles of P.V
    static constexpr bool EVEN_ODD = TPR >= 2;     // token order inside a 16-token tile
    // Resident CTAs per SM: 1 for the wide layout (3 stages of 54 KB), 3 for
    // int4 D = 128 (shared memory: 4 stages of 18 KB each) and for int8, 4 for
    // int4 D = 64 (whose stages are half as large), 2 for D = 256.
    static constexpr int MIN_CTAS = WIDE ? 1 : ((D == 256) ? 2 : ((D == 128 || BITS == 8) ? 3 : 4));
    static_assert(BPT <= 128 || BPT == 256, "a token's codes span one 128-byte swizzle row or two blocks");
    static_assert(CODE_BYTES % 1024 == 0, "code tiles must keep the 1024-byte swizzle period");
    static_assert(STAGES * STAGE_BYTES >= NWC * 8 * D * 4, "merge buffer must fit in the stages");
};

// Token (within a 16-token tile) held by fragment row m.  For D <= 128 rows
// 0..7 take the even tokens and rows 8..15 the odd ones, so that the eight
// rows of every ldmatrix fall into eight different 16-byte bank groups of the
// swizzled tile and a C-fragment row pair (m, m+8) is two adjacent tokens.
// Merge-buffer layout: element d of head h = 2 tig + hh is stored at h * D +
// (d ^ merge_xor(tig)), which spreads the four tig lanes of each store over
// different banks (int4 rows d = 32s + 4gid + 2j: flip bits 0-1; int8 rows
// d = 16i + 2gid: flip bit 0 and bit 4).
template <int BITS>
__device__ __forceinline__ int merge_xor(int tig) {
    if constexpr (BITS == 8) return (tig & 1) | ((tig >> 1) << 4);
    else return tig;
}

template <class C>
__device__ __forceinline__ int tok_of_row(int m) {
    if constexpr (C::EVEN_ODD) return m < 8 ? 2 * m : 2 * (m - 8) + 1;
    else return m;
}

// Shared address of 16-byte segment `seg` of token `tok` in a code tile laid
// out by TMA boxes of 128-byte rows with CU_TENSOR_MAP_SWIZZLE_128B (segment
// seg of a 256-byte row sits in column block seg / 8).
template <class C>
__device__ __forceinline__ uint32_t code_addr(uint32_t tile, int tok, int seg) {
    const int half = seg / C::SPR, s = seg % C::SPR;
    const int row = tok / C::TPR;
    const int chunk = (tok % C::TPR) * C::SPR + s;
    return tile + half * C::HALF_BYTES + row * 128 + ((chunk ^ (row & 7)) << 4);
}

struct alignas(8) Half4 {
    __half2 a, b;
};

// NG fp16 values of one token row -> floats.
template <int NG>
__device__ __forceinline__ void load_row_sb(const uint16_t* base, int tok, float (&out)[NG]) {
    const uint16_t* p = base + tok * NG;
    if constexpr (NG == 1) {
        out[0] = __half2float(__ushort_as_half(p[0]));
    } else if constexpr (NG == 2) {
        const __half2 h = *reinterpret_cast<const __half2*>(p);
        out[0] = __low2float(h);
        out[1] = __high2float(h);
    } else {
        const Half4 h = *reinterpret_cast<const Half4*>(p);
        out[0] = __low2float(h.a);
        out[1] = __high2float(h.a);
        out[2] = __low2float(h.b);
        out[3] = __high2float(h.b);
    }
}

// NG fp16 values of two token rows; for D <= 128 the rows are adjacent and one
// load brings both.
template <class C, int NG>
__device__ __forceinline__ void load_pair_sb(const uint16_t* base, int tok_a, int tok_b, float (&a)[NG],
                                             float (&bb)[NG]) {
    if constexpr (C::EVEN_ODD && NG == 2) {  // tok_b == tok_a + 1
        const Half4 h = *reinterpret_cast<const Half4*>(base + tok_a * 2);
        a[0] = __low2float(h.a);
        a[1] = __high2float(h.a);
        bb[0] = __low2float(h.b);
        bb[1] = __high2float(h.b);
    } else if constexpr (C::EVEN_ODD && NG == 1) {
        const __half2 h = *reinterpret_cast<const __half2*>(base + tok_a);
        a[0] = __low2float(h);
        bb[0] = __high2float(h);
    } else {
        load_row_sb<NG>(base, tok_a, a);
        load_row_sb<NG>(base, tok_b, bb);
    }
}

__device__ __forceinline__ int clamp_len(const DecodeParams& p, const int32_t* src) {
    int len = __ldg(src);
    if (len < 0 || len > p.max_seq_len) {
        if (p.status != nullptr && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            atomicOr(p.status, TQ_DEV_SEQ_LEN);
        len = min(max(len, 0), p.max_seq_len);
    }
    return len;
}

// What the kernel writes (separate instantiations: an extra branch in the
// epilogue of the split kernel measured 0.45 us slower per 128K decode):
//  kOutParts    the run's partial state (m, l, acc), merged by the reduce;
//  kOutDirect   one run per sequence: fp16(acc / l) is the output;
//  kOutCluster  the runs of a (sequence, kv head) are one thread-block cluster
//               (n_splits <= 8 CTAs): the CTAs merge their states through
//               distributed shared memory and write the output, no reduce.
constexpr int kOutParts = 0, kOutDirect = 1, kOutCluster = 2;

template <int D, bool PAGED, int BITS, int OUT, bool WIDE>
__global__ void __launch_bounds__(Cfg<D, BITS, WIDE>::THREADS, Cfg<D, BITS, WIDE>::MIN_CTAS)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const DecodeParams p) {
    using C = Cfg<D, BITS, WIDE>;
    static_assert(!WIDE || wide_ok(D, BITS, PAGED), "the wide layout is for contiguous int4 head_dim 128");
    constexpr int NG = C::NG;
    __shared__ uint64_t full_bar[C::STAGES];
    __shared__ unsigned int done_cnt[C::STAGES];  // warps finished with the stage, cumulative
    __shared__ float mrg_m[C::NWC][8], mrg_l[C::NWC][8], mrg_t[C::NWC][8];
    // paged: the block-table entries of this run's pages, loaded once
    constexpr int kPageWindow = PAGED ? 256 : 1;
    __shared__ int32_t page_s[kPageWindow];
    // kOutCluster: this CTA's merged state, read by the cluster (acc after the
    // warps' merge buffer in the dynamic shared memory)
    constexpr int kClHeads = OUT == kOutCluster ? 8 : 1;
    __shared__ float cl_m[kClHeads], cl_l[kClHeads];
    extern __shared__ uint8_t dyn_smem[];
    const uint32_t dyn_base = smem_u32(dyn_smem);
    uint8_t* smem = dyn_smem + ((1024u - (dyn_base & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int32_t* len_src = p.seq_lens + b;
    if (p.wait_at_start == kWaitAtStart) pdl_wait_primary();
    if (p.order != nullptr) {
        // grids of several waves: the runs in the order the planning kernel
        // wrote (longest first), each run's kv heads consecutive; the entry
        // carries the sequence's (clamped, checked) length, read in parallel
        const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        const int2* e = p.order + lin / gridDim.y;
        const int item = __ldg(&e->x);
        len_src = &e->y;
        kvh = lin % gridDim.y;
        b = item / gridDim.x;
        split = item % gridDim.x;
    }
    const int G = p.group_q;
    const int len = clamp_len(p, len_src);
    const int t_begin = run_begin(split, p.units, p.n_splits, p.unit_tokens);
    const int t_end = min(run_begin(split + 1, p.units, p.n_splits, p.unit_tokens), len);
    const int n_tiles = t_end > t_begin ? (t_end - t_begin + C::T - 1) / C::T : 0;
    const long long row_base = (static_cast<long long>(b) * p.num_kv_heads + kvh) * p.capacity;  // contiguous

    int first_page = 0, n_win = 0;
    if constexpr (PAGED) {
        first_page = page_index(p.map, t_begin);
        n_win = t_end > t_begin ? page_index(p.map, t_end - 1) - first_page + 1 : 0;
        n_win = min(n_win, kPageWindow);
        for (int i = threadIdx.x; i < n_win; i += C::THREADS) {
            int pg = __ldg(p.map.block_table + static_cast<long long>(b) * p.map.max_pages + first_page + i);
            if (static_cast<unsigned>(pg) >= static_cast<unsigned>(p.map.num_pages)) {
                if (p.status != nullptr) atomicOr(p.status, TQ_DEV_PAGE);
                pg = 0;
            }
            page_s[i] = pg;
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            done_cnt[s] = 0;
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    // Rows the append of this step writes while this grid may already run
    // (programmatic dependent launch): a tile that uses any of them is issued
    // only after the append grid has completed.  Other tiles do not wait.
    int dep_lo = 0, dep_hi = 0;
    if (p.dep_write_pos != nullptr) {
        dep_lo = __ldg(p.dep_write_pos + b);
        dep_hi = dep_lo + p.dep_n_new;
    }

    // Fused append: rows [app_lo, app_hi) of this (b, kv head) are owned by
    // this run and quantized here before any tile that uses them is loaded.
    int app_lo = 0, app_hi = 0, app_wp = 0;
    if (p.app.n_new > 0) {
        const int wp = app_wp = __ldg(p.app.write_pos + b);
        if (wp < 0 || static_cast<long long>(wp) + p.app.n_new > p.capacity) {
            if (p.status != nullptr && threadIdx.x == 0 && split == 0 && kvh == 0)
                atomicOr(p.status, TQ_DEV_WRITE_POS);
        } else {
            const int own_end =
                split + 1 == p.n_splits ? p.capacity : run_begin(split + 1, p.units, p.n_splits, p.unit_tokens);
            app_lo = max(wp, run_begin(split, p.units, p.n_splits, p.unit_tokens));
            app_hi = min(wp + p.app.n_new, own_end);
        }
    }
    auto tile_uses = [&](int it, int lo, int hi) {
        const int t0 = t_begin + it * C::T;
        return lo < min(t0 + C::T, t_end) && hi > t0;
    };

    // Fill stage it % STAGES with tile it: both code tiles by TMA, the four
    // scale/bias rows by bulk copies; completion counted in bytes on full_bar.
    auto issue_tile = [&](int it, uint64_t policy) {
        const int stage = it % C::STAGES;
        const int t0 = t_begin + it * C::T;
        if (tile_uses(it, dep_lo, dep_hi)) pdl_wait_primary();
        // the tile's first row and its rows (a tile never crosses a page: pages hold whole tiles)
        long long row;
        int avail;
        if constexpr (PAGED) {
            const int pi = page_index(p.map, t0), w = pi - first_page;
            row = w < n_win ? (static_cast<long long>(page_s[w]) * p.num_kv_heads + kvh) * p.map.page_tokens +
                                  (t0 - pi * p.map.page_tokens)
                            : kv_row(p.map, p.num_kv_heads, b, kvh, t0, p.status);
            avail = C::T;
        } else {
            row = row_base + t0;
            avail = min(C::T, p.capacity - t0);  // rows left in this (b, kv head)
        }
        const uint32_t sb_bytes = static_cast<uint32_t>(avail) * NG * 2;
        uint8_t* st = smem + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full_bar[stage], 2 * C::CODE_BYTES + 4 * sb_bytes);
        if constexpr (C::HALVES == 1) {  // maps of 128-byte rows
            const int y = static_cast<int>((row * C::BPT) / 128);
            tma_load_2d(st, &tm_k, 0, y, &full_bar[stage], policy);
            tma_load_2d(st + C::CODE_BYTES, &tm_v, 0, y, &full_bar[stage], policy);
        } else {  // maps of BPT-byte rows, one box per 128-byte column block
            const int y = static_cast<int>(row);
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h) {
                tma_load_2d(st + h * C::HALF_BYTES, &tm_k, h * 128, y, &full_bar[stage], policy);
                tma_load_2d(st + C::CODE_BYTES + h * C::HALF_BYTES, &tm_v, h * 128, y, &full_bar[stage], policy);
            }
        }
        const long long sb_off = row * NG;
        uint8_t* sb = st + 2 * C::CODE_BYTES;
        bulk_load(sb + 0 * C::SB_BYTES, p.k_scale + sb_off, sb_bytes, &full_bar[stage], policy);
        bulk_load(sb + 1 * C::SB_BYTES, p.k_bias + sb_off, sb_bytes, &full_bar[stage], policy);
        bulk_load(sb + 2 * C::SB_BYTES, p.v_scale + sb_off, sb_bytes, &full_bar[stage], policy);
        bulk_load(sb + 3 * C::SB_BYTES, p.v_bias + sb_off, sb_bytes, &full_bar[stage], policy);
    };
    // The fused append, part 1: the first pass of new-row loads is issued
    // before the tile loads, so that it does not queue behind them in the
    // memory system (issued after them it made the owning CTA the last to
    // finish); its latency overlaps the tile and Q loads.
    const int app_tasks = (app_hi - app_lo) * NG * 2;  // eight lanes per (row, group, K|V)
    const int app_part = threadIdx.x & 7;
    // A row's 2 NG tasks are consecutive.  Up to head_dim 128 the K and V
    // tasks of a group are neighbours; at head_dim 256 the row's four K
    // groups come first, then its four V groups, so that each tensor's row
    // fills the 32 lanes of one warp (which its rotation spans).
    struct AppTask {
        int kv, g, r;
    };
    auto app_task = [&](int task) -> AppTask {
        if constexpr (NG == 4) return {(task >> 2) & 1, task & 3, app_lo + (task >> 3)};
        else return {task & 1, (task >> 1) % NG, app_lo + (task >> 1) / NG};
    };
    auto app_src = [&](int task) {
        const AppTask a = app_task(task);
        return (a.kv ? p.app.v_new : p.app.k_new) +
               (((static_cast<long long>(b) * p.num_kv_heads + kvh) * p.app.n_new + (a.r - app_wp)) * D +
                a.g * kGroup + app_part * 8);
    };
    uint4 app_raw = make_uint4(0, 0, 0, 0);
    if (static_cast<int>(threadIdx.x >> 3) < app_tasks)
        app_raw = __ldcs(reinterpret_cast<const uint4*>(app_src(threadIdx.x >> 3)));
    if (threadIdx.x == 0 && n_tiles > 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        const uint64_t policy = policy_evict_first();
        for (int it = 0; it < min(n_tiles, C::STAGES); ++it)
            if (!tile_uses(it, app_lo, app_hi)) issue_tile(it, policy);
    }

    // ------------------------------------------------------------ all warps
    const int gid = lane >> 2, tig = lane & 3;
    const float sl2 = p.score_scale_log2;

    // Q operands: head gid of the group (zero rows pad G up to 8).
    uint32_t qb[C::NKS][2];
    float qsum_own[NG];
    {
        const bool hv = gid < G;
        const uint16_t* qrow = p.q + (static_cast<long long>(b) * p.num_q_heads + kvh * G + (hv ? gid : 0)) * D;
        const __half sixteenth = __float2half_rn(0.0625f);
#pragma unroll
        for (int g = 0; g < NG; ++g) qsum_own[g] = 0.0f;
        // This lane's dims of head gid: E consecutive ones at E * tig in each
        // segment (int4: 32 dims, E = 8; int8: 16 dims, E = 4).
        constexpr int E = BITS == 8 ? 4 : 8;
        struct alignas(2 * E) QVec {
            __half h[E];
        };
        QVec qv[C::SPT];
#pragma unroll
        for (int s = 0; s < C::SPT; ++s) {
            if (hv) {
                qv[s] = *reinterpret_cast<const QVec*>(qrow + C::EPS * s + E * tig);
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) qv[s].h[j] = __ushort_as_half(0);
            }
        }
        if (p.rotate_q) {  // the same for the whole CTA
            // dim = 4E s + E tig + j: stages h < E in the lane, h = E, 2E across
            // the lanes of tig, then h = 4E, 8E, ... across the segments
            float v[C::SPT][E];
#pragma unroll
            for (int s = 0; s < C::SPT; ++s) {
#pragma unroll
                for (int j = 0; j < E; ++j) v[s][j] = __half2float(qv[s].h[j]);
                hadamard_in_lane<E>(v[s]);
            }
#pragma unroll
            for (int hl = 1; hl < 4; hl <<= 1) {
#pragma unroll
                for (int s = 0; s < C::SPT; ++s) hadamard_across_lanes<E>(v[s], lane, hl);
            }
#pragma unroll
            for (int hs = 1; hs < C::SPT; hs <<= 1) {
#pragma unroll
                for (int s = 0; s < C::SPT; ++s) {
                    if ((s & hs) != 0) continue;
#pragma unroll
                    for (int j = 0; j < E; ++j) {
                        const float u = v[s][j], w = v[s + hs][j];
                        v[s][j] = __fadd_rn(u, w);
                        v[s + hs][j] = __fsub_rn(u, w);
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < C::SPT; ++s) {
#pragma unroll
                for (int j = 0; j < E; ++j) qv[s].h[j] = __float2half_rn(__fmul_rn(v[s][j], p.rot_scale));
            }
        }
        if constexpr (BITS == 8) {
            // segment s = dims 16s .. 16s+15; k-step s: k=2tig,2tig+1 <- dims +4tig, +4tig+2;
            // k=2tig+8,+9 <- dims +4tig+1, +4tig+3 (bytes 0, 2 and 1, 3 of a register)
#pragma unroll
            for (int s = 0; s < C::SPT; ++s) {
                const __half* h = qv[s].h;
                qb[s][0] = pack_half2_bits(h[0], h[2]);
                qb[s][1] = pack_half2_bits(h[1], h[3]);
                qsum_own[(16 * s) / kGroup] +=
                    (__half2float(h[0]) + __half2float(h[1])) + (__half2float(h[2]) + __half2float(h[3]));
            }
        } else {
#pragma unroll
        for (int s = 0; s < C::SPT; ++s) {
            const __half* h = qv[s].h;
            // k-step (s,0): k=2tig,2tig+1 <- dims +0,+4 ; k=2tig+8,+9 <- dims +1,+5 (x 1/16)
            qb[2 * s][0] = pack_half2_bits(h[0], h[4]);
            qb[2 * s][1] = pack_half2_bits(__hmul(h[1], sixteenth), __hmul(h[5], sixteenth));
            // k-step (s,1): dims +2,+6 ; +3,+7 (x 1/16)
            qb[2 * s + 1][0] = pack_half2_bits(h[2], h[6]);
            qb[2 * s + 1][1] = pack_half2_bits(__hmul(h[3], sixteenth), __hmul(h[7], sixteenth));
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) part += __half2float(h[j]);
            qsum_own[(32 * s) / kGroup] += part;
        }
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            qsum_own[g] += __shfl_xor_sync(0xffffffffu, qsum_own[g], 1);
            qsum_own[g] += __shfl_xor_sync(0xffffffffu, qsum_own[g], 2);
        }
    }
    // bias coefficients for this thread's two C columns (heads 2tig, 2tig+1), log2 units
    float qs_l2[NG][2];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        qs_l2[g][0] = __shfl_sync(0xffffffffu, qsum_own[g], (2 * tig) * 4) * sl2;
        qs_l2[g][1] = __shfl_sync(0xffffffffu, qsum_own[g], (2 * tig + 1) * 4) * sl2;
    }
    const float k_coef = sl2 * 16777216.0f;  // undo the 2^-24 of the subnormal operands
    const int r0 = tok_of_row<C>(gid), r1 = tok_of_row<C>(gid + 8);

    float m_run[2] = {-INFINITY, -INFINITY};  // reference max of l, acc (lazy)
    float m_true[2] = {-INFINITY, -INFINITY}; // this thread's largest score so far
    // Per-lane state for its two heads (2tig, 2tig+1) as pairs, so that the
    // fp32 work runs on Blackwell's paired operations (__fadd2_rn and friends:
    // two independent round-to-nearest results, the same as two scalar ops).
    float2 l2 = make_float2(0.0f, 0.0f);       // sum of p
    float2 e2[NG];                             // sum of p * vbias (+ mean-code term) per group
    float2 acc2[C::NKS][2];                    // P.V code sums: [i][0] = C rows gid, [i][1] = rows gid + 8
#pragma unroll
    for (int g = 0; g < NG; ++g) e2[g] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < C::NKS; ++i) acc2[i][0] = acc2[i][1] = make_float2(0.0f, 0.0f);

    // The fused append, part 2: quantize the rows this run owns, publish them
    // to the async proxy, then load the first tiles that use them.
    if (app_lo < app_hi) {  // the same for the whole CTA
        static_assert((C::THREADS / 8) % (2 * NG) == 0, "a pass covers whole rows: a tensor's row starts a warp");
        for (int t0 = 0; t0 < app_tasks; t0 += C::THREADS / 8) {  // uniform trip count: shuffles inside
            const int task = t0 + (threadIdx.x >> 3);
            const bool valid = task < app_tasks;
            uint4 raw = app_raw;
            if (t0 > 0 && valid) raw = __ldcs(reinterpret_cast<const uint4*>(app_src(task)));
            if (p.app.flags != 0) {  // the same for the whole CTA: rows are stored rotated
                // A row's K (or V) sits in 8 NG lanes of one warp: element
                // 64 g + 8 part + j.  Stages h = 1, 2, 4 in the lane, h = 8, 16,
                // 32 across lane bits 0-2 (part), then h = 64 across lane bit 4
                // (g, head_dim 128: K and V interleaved) or h = 64, 128 across
                // lane bits 3 and 4 (g, head_dim 256).
                float v[8];
                halves_to_floats<8>(&raw, v);
                hadamard_in_lane<8>(v);
#pragma unroll
                for (int hl = 1; hl < 8; hl <<= 1) hadamard_across_lanes<8>(v, lane, hl);
                if constexpr (NG == 2) hadamard_across_lanes<8>(v, lane, 16);
                if constexpr (NG == 4) {
                    hadamard_across_lanes<8>(v, lane, 8);
                    hadamard_across_lanes<8>(v, lane, 16);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], p.app.rot_scale);
                uint4 rot;
                floats_to_halves<8>(v, &rot);
                if ((p.app.flags & (app_task(task).kv ? TQ_ROTATE_V : TQ_ROTATE_K)) != 0) raw = rot;
            }
            const GroupQ<BITS> gq = quantize_lane8<BITS>(raw);
            if (valid) {
                const AppTask a = app_task(task);
                const int kv = a.kv, g = a.g, r = a.r;
                long long row;
                if constexpr (PAGED) row = kv_row(p.map, p.num_kv_heads, b, kvh, r, p.status);
                else row = row_base + r;
                uint8_t* dst = (kv ? p.app.v_codes : p.app.k_codes) + row * C::BPT + g * (kGroup * BITS / 8) +
                               app_part * BITS;  // this lane's 8 codes: BITS bytes
                if constexpr (BITS == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(gq.codes[0], gq.codes[1]);
                else *reinterpret_cast<uint32_t*>(dst) = gq.codes[0];
                if (app_part == 0) {
                    (kv ? p.app.v_scale : p.app.k_scale)[row * NG + g] = __half_as_ushort(gq.scale);
                    (kv ? p.app.v_bias : p.app.k_bias)[row * NG + g] = __half_as_ushort(gq.bias);
                }
            }
        }
        // Ordering: the proxy fence makes the stores visible to later TMA /
        // bulk reads; the reads are issued after a CTA-scope synchronisation
        // with every writer -- the barrier below for the first STAGES tiles,
        // the per-stage release count (each warp's fence and counter update
        // after its stores) for a later refill.
        fence_proxy_async_global();
        bool early = false;
        for (int it = 0; it < min(n_tiles, C::STAGES); ++it) early |= tile_uses(it, app_lo, app_hi);
        if (early) {  // the same for the whole CTA
            __syncthreads();
            if (threadIdx.x == 0) {
                const uint64_t policy = policy_evict_first();
                for (int it = 0; it < min(n_tiles, C::STAGES); ++it)
                    if (tile_uses(it, app_lo, app_hi)) issue_tile(it, policy);
            }
        }
    }

    // ldmatrix row address pattern: lane -> (matrix, row)
    const int lm_mat = lane >> 3, lm_row = lane & 7;
    const int lm_tok = tok_of_row<C>((lm_mat & 1) * 8 + lm_row);  // token within the 16-token tile
    const int lm_seg = lm_mat >> 1;                                // first or second segment
    // per-lane ldmatrix offset inside a 16-token tile for each segment pair.
    // A tile starting at token tb begins at swizzle row tb / TPR; its phase
    // (that row mod 8) is XORed into the 16-byte chunk bits at use (always 0
    // for D >= 128, where a tile covers a multiple of 8 rows).
    uint32_t lm_off[C::SPT / 2];
#pragma unroll
    for (int sp = 0; sp < C::SPT / 2; ++sp) lm_off[sp] = code_addr<C>(0u, lm_tok, 2 * sp + lm_seg);

    for (int it = 0; it < n_tiles; ++it) {
        const int stage = it % C::STAGES;
        if (!mbar_wait_bounded(&full_bar[stage], (it / C::STAGES) & 1)) {
            // the fill never completed: report, stop consuming (no further
            // refills are issued, so the other warps give up the same way)
            if (p.status) atomicOr(p.status, TQ_DEV_TIMEOUT);
            break;
        }
        const int t0 = t_begin + it * C::T;
        const uint8_t* st = smem + stage * C::STAGE_BYTES;
        const uint32_t kc_s = smem_u32(st);
        const uint32_t vc_s = smem_u32(st + C::CODE_BYTES);
        const uint16_t* ks_s = reinterpret_cast<const uint16_t*>(st + 2 * C::CODE_BYTES);
        const uint16_t* kb_s = ks_s + C::SB_BYTES / 2;
        const uint16_t* vs_s = kb_s + C::SB_BYTES / 2;
        const uint16_t* vb_s = vs_s + C::SB_BYTES / 2;

        // Only the last tile of a run can be partial; full tiles take a copy of
        // the body without the masking selects.
        auto stage_body = [&](auto tail_tag) {
            constexpr bool kTail = decltype(tail_tag)::value;
            // ---- scores of this warp's m-tiles (log2 units)
            float sc[C::MT][4];
    #pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                const int tb = (warp * C::MT + mt) * 16;
                const uint32_t sw = static_cast<uint32_t>((tb / C::TPR) & 7) << 4;
                float cg[NG][4];
    #pragma unroll
                for (int g = 0; g < NG; ++g) cg[g][0] = cg[g][1] = cg[g][2] = cg[g][3] = 0.0f;
    #pragma unroll
                for (int sp = 0; sp < C::SPT / 2; ++sp) {
                    uint32_t x0, x1, x2, x3;
                    ldmatrix_x4(kc_s + tb * C::ROWB + (lm_off[sp] ^ sw), x0, x1, x2, x3);
    #pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int s = 2 * sp + e;
                        const int g = (C::EPS * s) / kGroup;
                        const uint32_t xa = e ? x2 : x0;  // rows 0..7
                        const uint32_t xb = e ? x3 : x1;  // rows 8..15
                        if constexpr (BITS == 8) {
                            // bytes 0, 2 -> k 2tig, 2tig+1; bytes 1, 3 -> k 2tig+8, 2tig+9
                            mma_16816(cg[g], xa & kByte, xb & kByte, (xa >> 8) & kByte, (xb >> 8) & kByte, qb[s][0],
                                      qb[s][1]);
                        } else {
                            mma_16816(cg[g], xa & kLoNib, xb & kLoNib, xa & kHiNib, xb & kHiNib, qb[2 * s][0],
                                      qb[2 * s][1]);
                            const uint32_t ya = xa >> 8, yb = xb >> 8;
                            mma_16816(cg[g], ya & kLoNib, yb & kLoNib, ya & kHiNib, yb & kHiNib, qb[2 * s + 1][0],
                                      qb[2 * s + 1][1]);
                        }
                    }
                }
                float ksa[NG], kba[NG], ksb[NG], kbb[NG];
                load_pair_sb<C, NG>(ks_s, tb + r0, tb + r1, ksa, ksb);
                load_pair_sb<C, NG>(kb_s, tb + r0, tb + r1, kba, kbb);
                const bool va = !kTail || t0 + tb + r0 < t_end, vb = !kTail || t0 + tb + r1 < t_end;
                float2 sa = make_float2(0.0f, 0.0f), sb = make_float2(0.0f, 0.0f);  // (head 2tig, 2tig+1)
    #pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const float2 qs = make_float2(qs_l2[g][0], qs_l2[g][1]);
                    const float ka = ksa[g] * k_coef, kb = ksb[g] * k_coef;
                    sa = __ffma2_rn(make_float2(ka, ka), make_float2(cg[g][0], cg[g][1]),
                                    __ffma2_rn(make_float2(kba[g], kba[g]), qs, sa));
                    sb = __ffma2_rn(make_float2(kb, kb), make_float2(cg[g][2], cg[g][3]),
                                    __ffma2_rn(make_float2(kbb[g], kbb[g]), qs, sb));
                }
                // masked rows may hold stale bits: select, never compute with them
                sc[mt][0] = va ? sa.x : -INFINITY;
                sc[mt][1] = va ? sa.y : -INFINITY;
                sc[mt][2] = vb ? sb.x : -INFINITY;
                sc[mt][3] = vb ? sb.y : -INFINITY;
            }

            // ---- online softmax update over this warp's tokens of the stage.
            // The running max only moves when a score exceeds it by more than
            // kLazyMax (log2 units): until then p = 2^(s - m) <= 2^kLazyMax,
            // harmless for the fp32 sums and the fp16 B operand, and the
            // cross-lane reduction and rescale are skipped for the stage.
            float mx[2];
            bool grow = false;
    #pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                mx[hh] = -INFINITY;
    #pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) mx[hh] = fmaxf(mx[hh], fmaxf(sc[mt][hh], sc[mt][2 + hh]));
                grow |= mx[hh] > m_run[hh] + kLazyMax;
                m_true[hh] = fmaxf(m_true[hh], mx[hh]);
            }
            if (__any_sync(0xffffffffu, grow)) {
    #pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float m = mx[hh];
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                    if (m > m_run[hh]) {
                        const float alpha = m_run[hh] == -INFINITY ? 0.0f : ex2_approx(m_run[hh] - m);
                        if (hh == 0) {
                            l2.x *= alpha;
    #pragma unroll
                            for (int g = 0; g < NG; ++g) e2[g].x *= alpha;
    #pragma unroll
                            for (int i = 0; i < C::NKS; ++i) {
                                acc2[i][0].x *= alpha;
                                acc2[i][1].x *= alpha;
                            }
                        } else {
                            l2.y *= alpha;
    #pragma unroll
                            for (int g = 0; g < NG; ++g) e2[g].y *= alpha;
    #pragma unroll
                            for (int i = 0; i < C::NKS; ++i) {
                                acc2[i][0].y *= alpha;
                                acc2[i][1].y *= alpha;
                            }
                        }
                        m_run[hh] = m;
                    }
                }
            }
            float m_use[2];
    #pragma unroll
            for (int hh = 0; hh < 2; ++hh) m_use[hh] = m_run[hh] == -INFINITY ? 0.0f : m_run[hh];

            // ---- P.V.  B operand r_t = p_t * vscale_tg rounded to fp16.  Its
            // rounding error e_t = r_t - fp16(r_t) (up to 2^-11 relative) meets
            // codes n in 0..15 whose mean is near 7.5, so sum_t e_t n_t would
            // be a visible bias next to the small attention output at long
            // context.  Most of it is the mean part 7.5 * sum_t e_t, which is
            // added back in fp32 together with the bias term; what is left,
            // sum_t e_t (n_t - 7.5), is at most half as large and averages out.
            uint32_t bhi[C::MT][NG][2];
    #pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                const int tb = (warp * C::MT + mt) * 16;
                const bool va = !kTail || t0 + tb + r0 < t_end, vb = !kTail || t0 + tb + r1 < t_end;
                const float2 nm = make_float2(-m_use[0], -m_use[1]);
                const float2 da = __fadd2_rn(make_float2(sc[mt][0], sc[mt][1]), nm);
                const float2 db = __fadd2_rn(make_float2(sc[mt][2], sc[mt][3]), nm);
                const float2 pa = make_float2(ex2_approx(da.x), ex2_approx(da.y));  // rows a, heads (2tig, 2tig+1)
                const float2 pb = make_float2(ex2_approx(db.x), ex2_approx(db.y));  // rows b
                l2 = __fadd2_rn(l2, __fadd2_rn(pa, pb));
                float vsa[NG], vba[NG], vsb[NG], vbb[NG];
                load_pair_sb<C, NG>(vs_s, tb + r0, tb + r1, vsa, vsb);
                load_pair_sb<C, NG>(vb_s, tb + r0, tb + r1, vba, vbb);
    #pragma unroll
                for (int g = 0; g < NG; ++g) {
                    // masked rows may hold stale scale/bias bits: select, never multiply
                    const float sa = va ? vsa[g] : 0.0f, sb = vb ? vsb[g] : 0.0f;
                    const float ba = va ? vba[g] : 0.0f, bb = vb ? vbb[g] : 0.0f;
                    const float2 q01 = __fmul2_rn(pa, make_float2(sa, sa)), q23 = __fmul2_rn(pb, make_float2(sb, sb));
                    const __half2 h01 = __float22half2_rn(q01), h23 = __float22half2_rn(q23);
                    const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                    const float2 m1 = make_float2(-1.0f, -1.0f);
                    e2[g] = __ffma2_rn(pa, make_float2(ba, ba), __ffma2_rn(pb, make_float2(bb, bb), e2[g]));
                    const float2 r = __fadd2_rn(__ffma2_rn(f01, m1, q01), __ffma2_rn(f23, m1, q23));  // q - fp16(q)
                    e2[g] = __ffma2_rn(make_float2(C::CODE_MEAN, C::CODE_MEAN), r, e2[g]);
                    bhi[mt][g][0] = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&h01));
                    bhi[mt][g][1] = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&h23));
                }
            }
            // The stage's sum_t r_t n_t (all MT tiles) goes into fresh tensor-core
            // accumulators and is then added to the running state with
            // round-to-nearest fp32 adds.  The code sum is ~7.5 sum_t r_t while the
            // attention output is what is left after the bias term cancels most
            // of it, so a long chain of tensor-core accumulations (whose fp32 sums
            // are not round-to-nearest) would leave a systematic error far above
            // 1e-3 of the output at long context.
    #pragma unroll
            for (int sp = 0; sp < C::SPT / 2; ++sp) {
                uint32_t x[C::MT][4];
    #pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    const int tb = (warp * C::MT + mt) * 16;
                    const uint32_t sw = static_cast<uint32_t>((tb / C::TPR) & 7) << 4;
                    ldmatrix_x4_trans(vc_s + tb * C::ROWB + (lm_off[sp] ^ sw), x[mt][0], x[mt][1], x[mt][2], x[mt][3]);
                }
    #pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int s = 2 * sp + e;
                    const int g = (C::EPS * s) / kGroup;
                    if constexpr (BITS == 8) {
                        // A = V^T: low bytes -> dims 16s + 2gid (rows 0..7), high bytes ->
                        // dims 16s + 2gid + 1 (rows 8..15); tokens in k
                        float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    #pragma unroll
                        for (int mt = 0; mt < C::MT; ++mt) {
                            const uint32_t xa = e ? x[mt][2] : x[mt][0];  // tokens of rows 0..7  (k 0..7)
                            const uint32_t xb = e ? x[mt][3] : x[mt][1];  // tokens of rows 8..15 (k 8..15)
                            mma_16816(t, xa & kByte, (xa >> 8) & kByte, xb & kByte, (xb >> 8) & kByte,
                                      bhi[mt][g][0], bhi[mt][g][1]);
                        }
                        acc2[s][0] = __fadd2_rn(acc2[s][0], make_float2(t[0], t[1]));
                        acc2[s][1] = __fadd2_rn(acc2[s][1], make_float2(t[2], t[3]));
                    } else {
    #pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    #pragma unroll
                        for (int mt = 0; mt < C::MT; ++mt) {
                            const uint32_t xa = e ? x[mt][2] : x[mt][0];  // tokens of rows 0..7  (k 0..7)
                            const uint32_t xb = e ? x[mt][3] : x[mt][1];  // tokens of rows 8..15 (k 8..15)
                            const uint32_t ua = j ? (xa >> 8) : xa, ub = j ? (xb >> 8) : xb;
                            const uint32_t a0 = ua & kLoNib, a1 = ua & kHiNib, a2 = ub & kLoNib, a3 = ub & kHiNib;
                            mma_16816(t, a0, a1, a2, a3, bhi[mt][g][0], bhi[mt][g][1]);
                        }
                        acc2[2 * s + j][0] = __fadd2_rn(acc2[2 * s + j][0], make_float2(t[0], t[1]));
                        acc2[2 * s + j][1] = __fadd2_rn(acc2[2 * s + j][1], make_float2(t[2], t[3]));
                    }
                    }
                }
            }
        };
        if (t0 + C::T <= t_end) stage_body(std::false_type{});
        else stage_body(std::true_type{});

        // Release the stage.  The last warp to finish it refills it with tile
        // it + STAGES: its fence orders every warp's reads of the stage (made
        // visible by their fences before the counter update) before the
        // asynchronous copies that overwrite it.
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const unsigned int before = atomicAdd(&done_cnt[stage], 1u);
            if (before % C::NWC == C::NWC - 1 && it + C::STAGES < n_tiles) {
                __threadfence_block();
                fence_proxy_async_shared();
                issue_tile(it + C::STAGES, policy_evict_first());
            }
        }
    }

    // back to per-head scalars for the epilogue
    float l_run[2] = {l2.x, l2.y};
    float e_run[NG][2];
    float acc[C::NKS][4];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        e_run[g][0] = e2[g].x;
        e_run[g][1] = e2[g].y;
    }
#pragma unroll
    for (int i = 0; i < C::NKS; ++i) {
        acc[i][0] = acc2[i][0].x;
        acc[i][1] = acc2[i][0].y;
        acc[i][2] = acc2[i][1].x;
        acc[i][3] = acc2[i][1].y;
    }

    // ---- reduce per-thread sums and maxima over the 8 token rows (lanes differing in gid)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) m_true[hh] = fmaxf(m_true[hh], __shfl_xor_sync(0xffffffffu, m_true[hh], off));
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], off);
#pragma unroll
            for (int g = 0; g < NG; ++g) e_run[g][hh] += __shfl_xor_sync(0xffffffffu, e_run[g][hh], off);
        }
    }

    // ---- merge the consumer warps' states through shared memory
    // (every issued fill has been waited for by every warp once all pass this barrier)
    __syncthreads();
    float* mrg_acc = reinterpret_cast<float*>(smem);  // [NWC][8][D]
    float* cl_acc = mrg_acc + C::NWC * 8 * D;          // kOutCluster: [8][D]
    static_assert(OUT != kOutCluster || C::STAGES * C::STAGE_BYTES >= (C::NWC + 1) * 8 * D * 4,
                  "the cluster state must fit in the stages after the merge buffer");
    {
        float* wacc = mrg_acc + warp * 8 * D;
        if constexpr (BITS == 8) {
#pragma unroll
            for (int i = 0; i < C::NKS; ++i) {
                const int d_lo = 16 * i + 2 * gid;  // fragment row gid (low bytes)
                const int d_hi = d_lo + 1;          // fragment row gid + 8 (high bytes)
                const int g = d_lo / kGroup;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int h = 2 * tig + hh, x = merge_xor<BITS>(tig);
                    wacc[h * D + (d_lo ^ x)] = fmaf(acc[i][hh], 16777216.0f, e_run[g][hh]);
                    wacc[h * D + (d_hi ^ x)] = fmaf(acc[i][2 + hh], 16777216.0f, e_run[g][hh]);
                }
            }
        } else {
#pragma unroll
        for (int i = 0; i < C::NKS; ++i) {
            const int s = i >> 1, j = i & 1;
            const int d_lo = 32 * s + 4 * gid + 2 * j;  // fragment row gid
            const int d_hi = d_lo + 1;                  // fragment row gid + 8 (x16 operand)
            const int g = d_lo / kGroup;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                // element d of head h sits at h * D + (d ^ (h >> 1 & 3)): the XOR
                // spreads the four tig lanes of a store over different banks
                const int h = 2 * tig + hh;
                wacc[h * D + (d_lo ^ tig)] = fmaf(acc[i][hh], 16777216.0f, e_run[g][hh]);
                wacc[h * D + (d_hi ^ tig)] = fmaf(acc[i][2 + hh], 1048576.0f, e_run[g][hh]);
            }
        }
        }
        if (gid == 0) {
            mrg_m[warp][2 * tig] = m_run[0];
            mrg_m[warp][2 * tig + 1] = m_run[1];
            mrg_t[warp][2 * tig] = m_true[0];
            mrg_t[warp][2 * tig + 1] = m_true[1];
            mrg_l[warp][2 * tig] = l_run[0];
            mrg_l[warp][2 * tig + 1] = l_run[1];
        }
    }
    __syncthreads();
    const float ln2 = 0.69314718055994531f;
    for (int idx = threadIdx.x; idx < G * D; idx += C::NWC * 32) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NWC; ++w) M = fmaxf(M, mrg_t[w][h]);  // the run's largest score
        float L = 0.0f, A = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::NWC; ++w) {
                const float wt = mrg_m[w][h] == -INFINITY ? 0.0f : ex2_approx(mrg_m[w][h] - M);
                L = fmaf(wt, mrg_l[w][h], L);
                A = fmaf(wt, mrg_acc[(w * 8 + h) * D + (d ^ merge_xor<BITS>(h >> 1 & 3))], A);
            }
        }
        const long long ph = (static_cast<long long>(b) * p.num_q_heads + kvh * G + h) * p.n_splits + split;
        if constexpr (OUT == kOutDirect) {  // one run: the same division and rounding as the reduce of one part
            p.out[ph * D + d] = __half_as_ushort(__float2half_rn(L > 0.0f ? __fdiv_rn(A, L) : 0.0f));
        } else if constexpr (OUT == kOutCluster) {  // the partial state, kept for the cluster merge below
            cl_acc[h * D + d] = A;
            if (d == 0) {
                cl_m[h] = M == -INFINITY ? -INFINITY : M * ln2;
                cl_l[h] = L;
            }
        } else {
            p.part_acc[ph * D + d] = A;
            if (d == 0) {
                p.part_m[ph] = M == -INFINITY ? -INFINITY : M * ln2;
                p.part_l[ph] = L;
            }
        }
    }
    if constexpr (OUT == kOutCluster) {
        // Merge the cluster's partial states (one per run of this sequence and
        // kv head, read from the runs' shared memory), each CTA taking a share
        // of the (head, dim) outputs, with the reduce kernel's arithmetic for
        // up to eight parts, operation for operation: M = max of m over parts
        // with l > 0, w = expf(m - M), L = the reduce's shuffle-tree sum of
        // fmaf(w, l, 0) (lanes 0..7: ((0 + 4) + (2 + 6)) + ((1 + 5) + (3 + 7))),
        // the output sum of fmaf(w, acc, 0) in part order, fp16(acc / L).  The
        // result is bit for bit the one of phase 1 with partials plus the reduce.
        cluster_sync();
        const int n_runs = static_cast<int>(gridDim.x), rank = static_cast<int>(cluster_ctarank());
        for (int idx = rank * C::THREADS + threadIdx.x; idx < G * D; idx += n_runs * C::THREADS) {
            const int h = idx / D, d = idx % D;
            // all the runs' values in one round trip of remote loads
            float m[kMaxClusterRuns], w[kMaxClusterRuns], v[kMaxClusterRuns], a[kMaxClusterRuns];
#pragma unroll
            for (int r = 0; r < kMaxClusterRuns; ++r) {
                v[r] = r < n_runs ? ld_cluster_f32(&cl_l[h], r) : 0.0f;
                m[r] = r < n_runs ? ld_cluster_f32(&cl_m[h], r) : -INFINITY;
                a[r] = r < n_runs ? ld_cluster_f32(&cl_acc[h * D + d], r) : 0.0f;
            }
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < kMaxClusterRuns; ++r) {
                if (!(v[r] > 0.0f)) m[r] = -INFINITY;  // empty parts carry no weight
                M = fmaxf(M, m[r]);
            }
#pragma unroll
            for (int r = 0; r < kMaxClusterRuns; ++r) {
                w[r] = m[r] == -INFINITY ? 0.0f : expf(m[r] - M);
                v[r] = fmaf(w[r], v[r], 0.0f);
            }
            const float L = ((v[0] + v[4]) + (v[2] + v[6])) + ((v[1] + v[5]) + (v[3] + v[7]));
            float t = 0.0f;
#pragma unroll
            for (int r = 0; r < kMaxClusterRuns; ++r) t += w[r] != 0.0f ? fmaf(w[r], a[r], 0.0f) : 0.0f;
            const long long o = (static_cast<long long>(b) * p.num_q_heads + kvh * G + h) * D + d;
            p.out[o] = __half_as_ushort(__float2half_rn(L > 0.0f ? __fdiv_rn(t, L) : 0.0f));
        }
        cluster_sync();  // no CTA leaves while another may still read its shared memory
    }
}

template <int D, bool PAGED, int BITS, int OUT, bool WIDE>
cudaError_t set_smem_attr() {
    // per device; setting the attribute twice (two host threads) is harmless
    static std::atomic<bool> done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, PAGED, BITS, OUT, WIDE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, BITS, WIDE>::SMEM_BYTES);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
    return e;
}

template <int D, bool PAGED, int BITS, int OUT, bool WIDE>
cudaError_t launch_mode(cudaLaunchConfig_t& cfg, const DecodeParams& p, const CUtensorMap& tm_k,
                        const CUtensorMap& tm_v) {
    const cudaError_t e = set_smem_attr<D, PAGED, BITS, OUT, WIDE>();
    if (e != cudaSuccess) return e;
    cfg.blockDim = dim3(Cfg<D, BITS, WIDE>::THREADS);
    cfg.dynamicSmemBytes = Cfg<D, BITS, WIDE>::SMEM_BYTES;
    return cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, PAGED, BITS, OUT, WIDE>, tm_k, tm_v, p);
}

template <int D, bool PAGED, int BITS, bool WIDE>
cudaError_t launch_out(cudaLaunchConfig_t& cfg, const DecodeParams& p, const CUtensorMap& tm_k,
                       const CUtensorMap& tm_v, int out) {
    if (out == kOutDirect) return launch_mode<D, PAGED, BITS, kOutDirect, WIDE>(cfg, p, tm_k, tm_v);
    if (out == kOutCluster) return launch_mode<D, PAGED, BITS, kOutCluster, WIDE>(cfg, p, tm_k, tm_v);
    return launch_mode<D, PAGED, BITS, kOutParts, WIDE>(cfg, p, tm_k, tm_v);
}

// p.out set: the kernel writes the output itself, one run per sequence
// (n_splits = 1) or the runs of each (sequence, kv head) as one cluster.
template <int D, int BITS>
cudaError_t launch_d(const DecodeParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v, cudaStream_t stream,
                     bool pdl_secondary) {
    const bool paged = p.map.block_table != nullptr;
    const int out = p.out == nullptr ? kOutParts : (p.n_splits == 1 ? kOutDirect : kOutCluster);
    if (out == kOutCluster && p.n_splits > kMaxClusterRuns) return cudaErrorInvalidValue;
    if (p.wide && !wide_ok(D, BITS, paged)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_splits, p.num_kv_heads, p.batch);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned int n = 0;
    if (pdl_secondary) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (out == kOutCluster) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned int>(p.n_splits);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    if (paged) return launch_out<D, true, BITS, false>(cfg, p, tm_k, tm_v, out);
    if constexpr (wide_ok(D, BITS, false)) {
        if (p.wide) return launch_out<D, false, BITS, true>(cfg, p, tm_k, tm_v, out);
    }
    return launch_out<D, false, BITS, false>(cfg, p, tm_k, tm_v, out);
}

// Clusters of n CTAs of the cluster-merging instantiation the device holds at
// once (0 if it cannot place one).
template <int D, bool PAGED, int BITS, bool WIDE>
int max_clusters_d(int n) {
    using C = Cfg<D, BITS, WIDE>;
    if (set_smem_attr<D, PAGED, BITS, kOutCluster, WIDE>() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned int>(n), 1, 1);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = static_cast<unsigned int>(n);
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, decode_mma_kernel<D, PAGED, BITS, kOutCluster, WIDE>, &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters;
}

template <int D, bool PAGED, int BITS, bool WIDE>
int ctas_per_sm_d() {
    using C = Cfg<D, BITS, WIDE>;
    if (set_smem_attr<D, PAGED, BITS, kOutParts, WIDE>() != cudaSuccess) return 1;
    int n = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<D, PAGED, BITS, kOutParts, WIDE>, C::THREADS,
                                                  C::SMEM_BYTES);
    return n > 0 ? n : 1;
}

}  // namespace

// (head_dim, bits) pairs with a kernel: int4 at 64 / 128 / 256, int8 at 64 / 128
// (an int8 row of 256 would not fit one 128-byte swizzle row).
bool mma_supported(int head_dim, int bits) {
    return (bits == 4 || bits == 8) && (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

#define TQ_DISPATCH(EXPR64_4, EXPR128_4, EXPR256_4, EXPR64_8, EXPR128_8, EXPR256_8, FALLBACK) \
    if (bits == 8) {                                                              \
        if (head_dim == 64) return EXPR64_8;                                      \
        if (head_dim == 128) return EXPR128_8;                                    \
        if (head_dim == 256) return EXPR256_8;                                    \
    } else {                                                                      \
        if (head_dim == 64) return EXPR64_4;                                      \
        if (head_dim == 128) return EXPR128_4;                                    \
        if (head_dim == 256) return EXPR256_4;                                    \
    }                                                                             \
    return FALLBACK;

int mma_tile_tokens(int head_dim, int bits, bool wide) {
    if (wide) return head_dim == 128 && bits == 4 ? Cfg<128, 4, true>::T : 0;
    TQ_DISPATCH(Cfg<64>::T, Cfg<128>::T, Cfg<256>::T, (Cfg<64, 8>::T), (Cfg<128, 8>::T), (Cfg<256, 8>::T), 0)
}

int mma_smem_bytes(int head_dim, int bits, bool wide) {
    if (wide) return head_dim == 128 && bits == 4 ? Cfg<128, 4, true>::SMEM_BYTES : 0;
    TQ_DISPATCH(Cfg<64>::SMEM_BYTES, Cfg<128>::SMEM_BYTES, Cfg<256>::SMEM_BYTES, (Cfg<64, 8>::SMEM_BYTES),
                (Cfg<128, 8>::SMEM_BYTES), (Cfg<256, 8>::SMEM_BYTES), 0)
}

bool mma_wide_supported(int head_dim, int bits, bool paged) { return wide_ok(head_dim, bits, paged); }

int mma_max_active_clusters(int head_dim, int bits, bool paged, bool wide, int n) {
    if (n < 2 || n > kMaxClusterRuns) return 0;
    if (wide) return wide_ok(head_dim, bits, paged) ? max_clusters_d<128, false, 4, true>(n) : 0;
    if (paged) {
        TQ_DISPATCH((max_clusters_d<64, true, 4, false>(n)), (max_clusters_d<128, true, 4, false>(n)),
                    (max_clusters_d<256, true, 4, false>(n)), (max_clusters_d<64, true, 8, false>(n)),
                    (max_clusters_d<128, true, 8, false>(n)), (max_clusters_d<256, true, 8, false>(n)), 0)
    }
    TQ_DISPATCH((max_clusters_d<64, false, 4, false>(n)), (max_clusters_d<128, false, 4, false>(n)),
                (max_clusters_d<256, false, 4, false>(n)), (max_clusters_d<64, false, 8, false>(n)),
                (max_clusters_d<128, false, 8, false>(n)), (max_clusters_d<256, false, 8, false>(n)), 0)
}

int mma_ctas_per_sm(int head_dim, int bits, bool wide) {
    if (wide) return head_dim == 128 && bits == 4 ? ctas_per_sm_d<128, false, 4, true>() : 1;
    TQ_DISPATCH((ctas_per_sm_d<64, false, 4, false>()), (ctas_per_sm_d<128, false, 4, false>()),
                (ctas_per_sm_d<256, false, 4, false>()), (ctas_per_sm_d<64, false, 8, false>()),
                (ctas_per_sm_d<128, false, 8, false>()), (ctas_per_sm_d<256, false, 8, false>()), 1)
}

cudaError_t launch_decode_mma(const DecodeParams& p, int head_dim, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                              cudaStream_t stream, bool pdl_secondary) {
    const int bits = p.bits;
    TQ_DISPATCH((launch_d<64, 4>(p, tm_k, tm_v, stream, pdl_secondary)),
                (launch_d<128, 4>(p, tm_k, tm_v, stream, pdl_secondary)),
                (launch_d<256, 4>(p, tm_k, tm_v, stream, pdl_secondary)),
                (launch_d<64, 8>(p, tm_k, tm_v, stream, pdl_secondary)),
                (launch_d<128, 8>(p, tm_k, tm_v, stream, pdl_secondary)),
                (launch_d<256, 8>(p, tm_k, tm_v, stream, pdl_secondary)), cudaErrorInvalidValue)
}

#undef TQ_DISPATCH

}  // namespace tq

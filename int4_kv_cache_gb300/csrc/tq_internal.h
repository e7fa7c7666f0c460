// tq_internal.h -- launch parameters shared by the C-ABI layer and kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "tq.h"

namespace tq {

constexpr int kGroup = 64;

// Where row t of (sequence b, kv head h) lives: in page P of the pool,
// row (P * num_kv_heads + h) * page_tokens + t % page_tokens, with P =
// block_table[b * max_pages + t / page_tokens].  A contiguous cache is the
// special case block_table = null, P = b, page_tokens = capacity.
struct RowMap {
    const int32_t* block_table;
    int32_t page_tokens, max_pages, num_pages;
    // paged maps: floor(t / page_tokens) = umulhi(t, page_magic) >> page_shift
    // for 0 <= t < 2^31 (set by with_page_divisor)
    uint32_t page_magic;
    int32_t page_shift;
};

// Division by the invariant page size as one multiply-high and a shift
// (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, round-up multiplier): with l = ceil(log2 d) and
// m = ceil(2^(31+l) / d) < 2^32, floor(t / d) = floor(t * m / 2^(31+l)) for
// every 0 <= t < 2^31, because m * d - 2^(31+l) < d <= 2^l makes the excess
// t * (m * d - 2^(31+l)) / (d * 2^(31+l)) smaller than 1/d.  Needs d >= 2.
inline RowMap with_page_divisor(RowMap m) {
    int l = 0;
    while ((1LL << l) < m.page_tokens) ++l;
    const unsigned long long d = static_cast<unsigned long long>(m.page_tokens);
    m.page_magic = static_cast<uint32_t>(((1ULL << (31 + l)) + d - 1) / d);
    m.page_shift = l - 1;
    return m;
}

// floor(n / d) for 0 <= n < 2^63 and 1 <= d < 2^31 by a 64-bit multiply-high
// and a shift: the same round-up multiplier with 63 in place of 31 (m =
// ceil(2^(63+l) / d) fits 64 bits and t * (m * d - 2^(63+l)) < 2^(63+l) for
// every n below 2^63); magic = 0 stands for d = 1.
struct FastDiv {
    uint64_t magic;
    int32_t shift;
    int32_t d;
};

inline FastDiv make_fastdiv(int32_t d) {
    FastDiv f{0, 0, d};
    if (d <= 1) return f;
    int l = 0;
    while ((1LL << l) < d) ++l;
    const unsigned __int128 num = static_cast<unsigned __int128>(1) << (63 + l);
    f.magic = static_cast<uint64_t>((num + static_cast<unsigned __int128>(d) - 1) / static_cast<unsigned>(d));
    f.shift = l - 1;
    return f;
}

#ifdef __CUDACC__
__device__ __forceinline__ long long fast_div(long long n, const FastDiv& f) {
    return f.magic == 0 ? n
                        : static_cast<long long>(__umul64hi(static_cast<unsigned long long>(n), f.magic) >> f.shift);
}

__device__ __forceinline__ int page_index(const RowMap& m, int t) {
    return static_cast<int>(__umulhi(static_cast<unsigned>(t), m.page_magic) >> m.page_shift);
}

__device__ __forceinline__ long long kv_row(const RowMap& m, int num_kv_heads, int b, int h, int t,
                                            int32_t* status) {
    int page = b, tp = t;
    if (m.block_table != nullptr) {
        const int pi = page_index(m, t);
        page = __ldg(m.block_table + static_cast<long long>(b) * m.max_pages + pi);
        tp = t - pi * m.page_tokens;
        if (static_cast<unsigned>(page) >= static_cast<unsigned>(m.num_pages)) {
            if (status != nullptr) atomicOr(status, TQ_DEV_PAGE);
            page = 0;
        }
    }
    return (static_cast<long long>(page) * num_kv_heads + h) * m.page_tokens + tp;
}
#endif

struct AppendParams {
    const uint16_t* k_new;    // [B][Hkv][n_new][D]
    const uint16_t* v_new;
    const int32_t* write_pos; // [B]
    uint8_t* k_codes;
    uint8_t* v_codes;
    uint16_t* k_scale;
    uint16_t* k_bias;
    uint16_t* v_scale;
    uint16_t* v_bias;
    int32_t* status;
    int32_t batch, num_kv_heads, head_dim, n_new, capacity;
    int32_t bits;      // code width: 4 or 8
    uint32_t flags;    // TQ_ROTATE_K / TQ_ROTATE_V: rotate the rows before quantizing them
    float rot_scale;   // fp32 value nearest 1 / sqrt(head_dim)
    RowMap map;
    // group index gi over [B][Hkv][n_new][NG] -> (row, g), (bh, i), (b, h)
    FastDiv div_ng, div_n_new, div_hkv;
};

// Geometry of one phase-1 launch: grid (n_splits, Hkv, B).  The sequence is
// cut into `units` units of `unit_tokens` tokens; CTA (s, kvh, b) covers units
// [floor(s * units / n_splits), floor((s + 1) * units / n_splits)) of sequence b
// (balanced runs), clipped to seq_lens[b].
struct DecodeParams {
    const uint16_t* q;        // [B][Hq][D]
    const int32_t* seq_lens;  // [B]
    const uint16_t* k_scale;  // [B][Hkv][cap][NG]
    const uint16_t* k_bias;
    const uint16_t* v_scale;
    const uint16_t* v_bias;
    const uint8_t* k_codes;   // [B][Hkv][cap][D/2] (the SIMT path reads these directly)
    const uint8_t* v_codes;
    float* part_m;            // [B][Hq][n_splits]   natural-log units
    float* part_l;            // [B][Hq][n_splits]
    float* part_acc;          // [B][Hq][n_splits][D]
    int32_t* status;          // optional device status word
    int32_t batch, num_q_heads, num_kv_heads, group_q;  // group_q = Hq / Hkv
    int32_t capacity, max_seq_len;
    int32_t unit_tokens, units, n_splits;
    float score_scale_log2;   // attn_scale * log2(e)
    // Set when the launch is a programmatic dependent of an append that wrote
    // rows [dep_write_pos[b], dep_write_pos[b] + dep_n_new): a tile that
    // uses any of them waits for the append before it is loaded.
    const int32_t* dep_write_pos;
    int32_t dep_n_new;
    RowMap map;
    // Fused append (tensor-core kernel only, app.n_new > 0): before reading
    // them, the CTA whose run owns rows [write_pos[b], write_pos[b] + n_new)
    // quantizes k_new / v_new into those rows itself.  A run owns
    // [run_begin(s), run_begin(s + 1)); the last run also owns the rows up to
    // the capacity.
    AppendParams app;
    int32_t bits;             // code width of the cache: 4 or 8
    // Keys stored rotated (tensor-core kernel only): the kernel attends with
    // fp16(rot_scale * H q), rotating each query head as it loads it.
    int32_t rotate_q;
    float rot_scale;
    // Where the kernel waits for the grid ahead of it on the stream (the
    // launch is always a programmatic dependent of that grid):
    //  kWaitAtStart    before its first read;
    //  kWaitForAppend  an append kernel is the grid ahead: only before the
    //                  tiles holding its rows (dep_write_pos).
    int32_t wait_at_start;
    // Optional dispatch order of the runs (grids of several waves): entry r
    // is {run b * n_splits + split, seq_lens[b] clamped to [0, max_seq_len]}
    // for CTA slots [r * Hkv, (r + 1) * Hkv) in launch order, one per kv head
    // (the length travels with the run so that a CTA makes one dependent read
    // before its first tile, not two).  Null: the grid's own order.
    const int2* order;
    // One run per sequence (n_splits = 1): the merged state is the output;
    // when set, the kernel writes fp16(acc / l) here instead of the partials.
    uint16_t* out;
    // The plan's SM layout: one 12-warp CTA per SM (mma_wide_supported only).
    int32_t wide;
};
constexpr int32_t kWaitForAppend = 0, kWaitAtStart = 1;
// Most rows per sequence the decode kernel appends itself; longer appends
// run the append kernel first.
constexpr int kFusedAppendMaxRows = 16;

// Longest-first dispatch order of the runs of a split decode (order.cu).
struct OrderParams {
    const int32_t* seq_lens;  // [B]
    int2* order;              // [B * n_splits] {run b * n_splits + s, clamped seq_lens[b]}, longest first
    int32_t* status;          // optional: TQ_DEV_SEQ_LEN for a length outside [0, max_seq_len]
    int32_t batch, max_seq_len, units, n_splits, unit_tokens, tile_tokens;
};

// Expansion of the cache into fp16 K/V [B][Hkv][n_rows][D] (comparison path).
struct DequantParams {
    const uint8_t* k_codes;
    const uint8_t* v_codes;
    const uint16_t* k_scale;
    const uint16_t* k_bias;
    const uint16_t* v_scale;
    const uint16_t* v_bias;
    uint16_t* k_out;
    uint16_t* v_out;
    int32_t batch, num_kv_heads, head_dim, capacity, n_rows, bits;
};

struct ReduceParams {
    const float* part_m;
    const float* part_l;
    const float* part_acc;
    uint16_t* out;            // [B][Hq][D]
    int32_t batch, num_q_heads, head_dim, n_parts;
    int32_t rotate_out;       // nonzero: out = H (merged output), for a cache whose V rows were rotated
    float rot_scale;
    // TQ_STEP_ADVANCE: after phase 1 has finished, seq_lens[b] and
    // write_pos[b] grow by adv_n (written once per sequence)
    int32_t* adv_seq_lens;
    int32_t* adv_write_pos;
    int32_t adv_n;
};


// Launchers (return the cudaError_t of the launch).
cudaError_t launch_quantize_append(const AppendParams& p, cudaStream_t stream);
// The same for large appends: a persistent grid (a few CTAs per SM of `sms`)
// streaming the fp16 rows through TMA.  tm_k / tm_v: k_new / v_new as
// [groups][128 bytes], boxes of kTmaAppendBoxRows rows, 128-byte swizzle.
constexpr long long kTmaAppendMinGroups = 8192;
constexpr int kTmaAppendCtasPerSm = 3;
constexpr int kTmaAppendBoxRows = 256;
cudaError_t launch_quantize_append_tma(const AppendParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                       int sms, cudaStream_t stream);
cudaError_t launch_decode_simt(const DecodeParams& p, int head_dim, cudaStream_t stream);
cudaError_t launch_decode_mma(const DecodeParams& p, int head_dim, const CUtensorMap& tm_k,
                              const CUtensorMap& tm_v, cudaStream_t stream, bool pdl_secondary);
// The append kernel, optionally letting the next launch start early (the
// decode kernel then waits only where it reads the appended rows).
cudaError_t launch_quantize_append_primary(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream, bool pdl_secondary);
cudaError_t launch_order_runs(const OrderParams& p, cudaStream_t stream);
cudaError_t launch_advance(int32_t* seq_lens, int32_t* write_pos, int batch, int n, cudaStream_t stream);
// The bounded-wait diagnostic (selftest.cu): *copied = sum of the 32-bit words
// of the 1 KB copied from src (0xFFFFFFFF if the copy did not land in time).
cudaError_t launch_wait_timeout_selftest(const void* src, int32_t* status, uint64_t limit_ns, uint32_t* copied,
                                         cudaStream_t stream);
cudaError_t launch_dequant(const DequantParams& p, int sm_count, cudaStream_t stream);
// out[r] = fp16(H x[r]) for rows of `dim` fp16 values (dim 64 / 128 / 256); out may be x.
cudaError_t launch_rotate_rows(const uint16_t* x, long long rows, int dim, uint16_t* out, float scale,
                               cudaStream_t stream);
// fp32 value nearest 1 / sqrt(dim), the rotation's normalisation.
inline float rotation_scale(int dim) { return static_cast<float>(1.0 / std::sqrt(static_cast<double>(dim))); }

// Tokens per pipeline stage of the tensor-core kernel (tiles are TMA boxes),
// for a code width of `bits` (4 or 8).
// wide: the layout of one 12-warp CTA per SM (contiguous int4 head_dim 128)
int mma_tile_tokens(int head_dim, int bits, bool wide);
int mma_smem_bytes(int head_dim, int bits, bool wide);
bool mma_wide_supported(int head_dim, int bits, bool paged);
bool mma_supported(int head_dim, int bits);
// Resident CTAs per SM of the phase-1 kernels (occupancy API).
int mma_ctas_per_sm(int head_dim, int bits, bool wide);
// Clusters of n (2..kMaxClusterRuns) CTAs of the cluster-merging phase-1
// kernel the device holds at once (occupancy API; 0: none).
int mma_max_active_clusters(int head_dim, int bits, bool paged, bool wide, int n);
int simt_ctas_per_sm(int head_dim);
// Largest n_parts the reduce kernel takes.
constexpr int kMaxReduceParts = 8192;
// Most runs per (sequence, kv head) merged inside phase 1 by a thread-block
// cluster (the portable cluster size); such launches write the output and
// need no reduce.
constexpr int kMaxClusterRuns = 8;
// Most CTAs a decode plan launches (bounds the workspace independently of the device).
constexpr int kMaxDecodeCtas = 2048;
// Tokens per work unit of the SIMT phase-1 kernel.
constexpr int kSimtTileTokens = 64;

// First token of run s of a phase-1 launch (runs are balanced over units).
__host__ __device__ inline int run_begin(int s, int units, int n_splits, int unit_tokens) {
    return static_cast<int>(static_cast<long long>(s) * units / n_splits) * unit_tokens;
}

// Decode (tensor-core phase 1 + reduce) with the partial states written to
// `partials` (partials_bytes long); TQ_ERR_WORKSPACE if they do not fit.
tq_status decode_into_partials(const tq_kv_cache* cache, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                               int32_t max_seq_len, float attn_scale, int32_t chunk, uint8_t* partials,
                               size_t partials_bytes, uint16_t* out, int32_t* status, cudaStream_t stream);
// Map a CUDA error to TQ_ERR_CUDA and remember it for tq_last_cuda_error().
tq_status record_cuda_status(cudaError_t e);

}  // namespace tq

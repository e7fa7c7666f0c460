// tq_api.cu -- the extern "C" boundary of libtq: argument checks, split-K
// planning, TMA descriptors and kernel dispatch.  No device allocation, no
// host synchronisation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "tq.h"
#include "tq_internal.h"

namespace {

thread_local int32_t g_last_cuda_error = 0;

tq_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return TQ_OK;
    g_last_cuda_error = static_cast<int32_t>(e);
    return TQ_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dim(int32_t d) { return d == 64 || d == 128 || d == 256; }

bool valid_impl(tq_impl impl) { return impl == TQ_IMPL_AUTO || impl == TQ_IMPL_MMA || impl == TQ_IMPL_SIMT; }

tq_status check_cache(const tq_kv_cache* c) {
    if (c == nullptr) return TQ_ERR_NULL;
    if (!c->k_codes || !c->v_codes || !c->k_scale || !c->k_bias || !c->v_scale || !c->v_bias) return TQ_ERR_NULL;
    if (c->batch < 1 || c->num_kv_heads < 1 || c->capacity < 16 || c->capacity % 16 != 0) return TQ_ERR_SHAPE;
    if (c->group_size != TQ_GROUP_SIZE || !supported_dim(c->head_dim)) return TQ_ERR_UNSUPPORTED;
    if (!tq::mma_supported(c->head_dim, c->bits)) return TQ_ERR_UNSUPPORTED;
    if (!aligned16(c->k_codes) || !aligned16(c->v_codes) || !aligned16(c->k_scale) || !aligned16(c->k_bias) ||
        !aligned16(c->v_scale) || !aligned16(c->v_bias))
        return TQ_ERR_ALIGN;
    // index arithmetic is 64-bit, but TMA row coordinates are int32
    const long long rows128 =
        static_cast<long long>(c->batch) * c->num_kv_heads * c->capacity * (c->head_dim * c->bits / 8) / 128;
    if (rows128 >= (1LL << 31)) return TQ_ERR_SHAPE;
    return TQ_OK;
}

// The cache as the kernels see it: the arrays, the sizes, and where each
// logical row lives (tq::RowMap).  A contiguous cache is one page per
// sequence; `capacity` is the logical capacity (max_pages * page_tokens when
// paged).  Field names follow tq_kv_cache so the code below reads the same
// for both layouts.
struct Store {
    uint8_t* k_codes;
    uint8_t* v_codes;
    uint16_t* k_scale;
    uint16_t* k_bias;
    uint16_t* v_scale;
    uint16_t* v_bias;
    int32_t batch, num_kv_heads, head_dim, group_size, capacity, bits;
    tq::RowMap map;
    bool paged;
};

// Sizes and pointers only (no checks): for planning queries.
Store shape_of(const tq_kv_cache* c) {
    Store st{};
    st.k_codes = c->k_codes;
    st.v_codes = c->v_codes;
    st.k_scale = c->k_scale;
    st.k_bias = c->k_bias;
    st.v_scale = c->v_scale;
    st.v_bias = c->v_bias;
    st.batch = c->batch;
    st.num_kv_heads = c->num_kv_heads;
    st.head_dim = c->head_dim;
    st.group_size = c->group_size;
    st.capacity = c->capacity;
    st.bits = c->bits;
    st.map = {nullptr, c->capacity, 1, c->batch, 0, 0};
    st.paged = false;
    return st;
}

tq_status store_of(const tq_kv_cache* c, Store* st) {
    tq_status s = check_cache(c);
    if (s != TQ_OK) return s;
    *st = shape_of(c);
    return TQ_OK;
}

// Pages hold whole pipeline tiles (128 tokens; 64 for head_dim 256), so a
// tile never crosses a page.
constexpr int kPageTokenMultiple = 128;

tq_status store_of(const tq_paged_kv_cache* c, Store* st) {
    if (c == nullptr) return TQ_ERR_NULL;
    if (!c->k_codes || !c->v_codes || !c->k_scale || !c->k_bias || !c->v_scale || !c->v_bias || !c->block_table)
        return TQ_ERR_NULL;
    if (c->batch < 1 || c->num_kv_heads < 1 || c->num_pages < 1 || c->max_pages_per_seq < 1) return TQ_ERR_SHAPE;
    if (c->page_tokens < kPageTokenMultiple || c->page_tokens % kPageTokenMultiple != 0) return TQ_ERR_SHAPE;
    if (c->group_size != TQ_GROUP_SIZE || !supported_dim(c->head_dim)) return TQ_ERR_UNSUPPORTED;
    if (!tq::mma_supported(c->head_dim, c->bits)) return TQ_ERR_UNSUPPORTED;
    if (!aligned16(c->k_codes) || !aligned16(c->v_codes) || !aligned16(c->k_scale) || !aligned16(c->k_bias) ||
        !aligned16(c->v_scale) || !aligned16(c->v_bias))
        return TQ_ERR_ALIGN;
    const long long cap = static_cast<long long>(c->max_pages_per_seq) * c->page_tokens;
    if (cap >= (1LL << 31)) return TQ_ERR_SHAPE;
    const long long rows128 =
        static_cast<long long>(c->num_pages) * c->num_kv_heads * c->page_tokens * (c->head_dim * c->bits / 8) / 128;
    if (rows128 >= (1LL << 31)) return TQ_ERR_SHAPE;
    Store& t = *st;
    t = Store{};
    t.k_codes = c->k_codes;
    t.v_codes = c->v_codes;
    t.k_scale = c->k_scale;
    t.k_bias = c->k_bias;
    t.v_scale = c->v_scale;
    t.v_bias = c->v_bias;
    t.batch = c->batch;
    t.num_kv_heads = c->num_kv_heads;
    t.head_dim = c->head_dim;
    t.group_size = c->group_size;
    t.capacity = static_cast<int32_t>(cap);
    t.bits = c->bits;
    t.map = tq::with_page_divisor({c->block_table, c->page_tokens, c->max_pages_per_seq, c->num_pages, 0, 0});
    t.paged = true;
    return TQ_OK;
}

// ---------------------------------------------------------------- TMA maps --
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// The code array of a cache as a 2-D uint8 tensor map for the decode kernel's
// tiles of `tile_tokens` tokens, with the 128-byte swizzle; reads past the end
// are zero-filled.
tq_status make_code_map(CUtensorMap* map, const uint8_t* codes, const Store* c, int tile_tokens) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return cuda_status(cudaErrorNotSupported);
    const cuuint64_t bpt = static_cast<cuuint64_t>(c->head_dim) * c->bits / 8;  // code bytes per token
    const cuuint64_t tokens = static_cast<cuuint64_t>(c->map.num_pages) * c->num_kv_heads * c->map.page_tokens;
    // Tokens of up to 128 bytes: the codes seen as rows of 128 bytes, a tile of
    // tile_tokens tokens one box.  256-byte tokens (int8, head_dim 256): rows of
    // 256 bytes, a tile two boxes of 128-byte columns.
    const bool wide = bpt > 128;
    cuuint64_t dims[2] = {wide ? bpt : 128, wide ? tokens : tokens * bpt / 128};
    cuuint64_t strides[1] = {wide ? bpt : 128};
    cuuint32_t box[2] = {128, static_cast<cuuint32_t>(wide ? tile_tokens : tile_tokens * bpt / 128)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_status(cudaErrorInvalidValue);
    return TQ_OK;
}

// A row-major array of `rows` rows of 128 bytes seen as uint8 [rows][128], boxes
// of `box_rows` rows with the 128-byte swizzle (the fp16 input of an append:
// one group of 64 halves per row).
tq_status make_rows_map(CUtensorMap* map, const void* base, unsigned long long rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return cuda_status(cudaErrorNotSupported);
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_status(cudaErrorInvalidValue);
    return TQ_OK;
}

// ------------------------------------------------------------ device facts --
struct DeviceFacts {
    int sms = 0;
    int mma_ctas[2][3] = {{0, 0, 0}, {0, 0, 0}};  // per code width (4, 8) and head_dim 64 / 128 / 256
    int wide_ctas = 0;  // the one-CTA-per-SM layout (contiguous int4, head_dim 128)
    int simt_ctas[3] = {0, 0, 0};
    // clusters of n CTAs of the cluster-merging kernel held at once, per code
    // width, head_dim, layout (contiguous, paged) and n
    int clusters[2][3][2][tq::kMaxClusterRuns + 1] = {};
    int wide_clusters[tq::kMaxClusterRuns + 1] = {};
};

int dim_index(int d) { return d == 64 ? 0 : (d == 128 ? 1 : 2); }

tq_status device_facts(DeviceFacts** out) {
    static DeviceFacts facts[64];
    static std::atomic<bool> ready[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= 64) return TQ_ERR_UNSUPPORTED;
    if (!ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[dev].load(std::memory_order_relaxed)) {
            DeviceFacts f;
            e = cudaDeviceGetAttribute(&f.sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return cuda_status(e);
            const int dims[3] = {64, 128, 256};
            for (int i = 0; i < 3; ++i) {
                f.mma_ctas[0][i] = tq::mma_ctas_per_sm(dims[i], 4, false);
                if (tq::mma_supported(dims[i], 8)) f.mma_ctas[1][i] = tq::mma_ctas_per_sm(dims[i], 8, false);
                f.simt_ctas[i] = tq::simt_ctas_per_sm(dims[i]);
                for (int bi = 0; bi < 2; ++bi) {
                    if (!tq::mma_supported(dims[i], bi ? 8 : 4)) continue;
                    for (int pg = 0; pg < 2; ++pg)
                        for (int n = 2; n <= tq::kMaxClusterRuns; ++n)
                            f.clusters[bi][i][pg][n] =
                                tq::mma_max_active_clusters(dims[i], bi ? 8 : 4, pg != 0, false, n);
                }
            }
            f.wide_ctas = tq::mma_ctas_per_sm(128, 4, true);
            for (int n = 2; n <= tq::kMaxClusterRuns; ++n)
                f.wide_clusters[n] = tq::mma_max_active_clusters(128, 4, false, true, n);
            cudaGetLastError();  // occupancy queries must leave no pending error
            facts[dev] = f;
            ready[dev].store(true, std::memory_order_release);
        }
    }
    *out = &facts[dev];
    return TQ_OK;
}

// ------------------------------------------------------------- decode plan --
struct Plan {
    int n_splits, unit_tokens, units;
    bool merged = false;  // the decode merges the runs itself (one run, or one cluster per sequence and kv head)
    int tile_tokens = 0;  // the kernel's pipeline tile
    long long resident = 0;  // CTAs the device holds at once for this kernel
    bool wide = false;    // one 12-warp CTA per SM (else several 4-warp CTAs)
    long long waves = 1;  // ceil(CTAs / resident)
};

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Balanced runs of whole units (the kernel's pipeline tile, or the chunk if
// that is smaller, so that runs cover the sequence evenly whatever its length
// in chunks), as many per (sequence, kv head) as minimise a model of the
// decode's time: waves x (longest run + a fixed cost per CTA), waves =
// ceil(CTAs / resident CTA slots), plus the reduce when one runs.  The fixed
// cost (pipeline fill, the query load, the partial-state store) is worth
// about two tiles of streaming, the reduce (the tail of the partial states'
// round trip; its launch overlaps phase 1) about one: on a GB300 the Gemma
// shape at 950 tokens decodes in 7.3 us as 8 merged runs of two tiles and in
// 7.5 us as 15 runs of one tile + the reduce, and at 2,048 tokens in 8.8 us
// as 16 runs of two tiles + the reduce against 9.6 us as 8 merged runs.  With `merge` (the decode may merge the runs
// itself), one run per sequence, or up to kMaxClusterRuns runs in a grid of
// one wave (one thread-block cluster per sequence and kv head), needs no
// reduce.  Within one wave count more runs are shorter, so the candidates are
// the largest run count of each wave count, the largest that phase 1 can
// merge, and one run, each taken down to the fewest runs with the same
// longest run; ties keep the fewer runs.  One sequence of 128K fills the
// resident slots once (57 runs with 8 kv heads and 456 slots); a batch whose
// grid needs several waves gets a CTA count just under a whole number of
// waves (16 sequences of 32K: 7 runs, 896 CTAs for 912 slots: 110 us against
// 141 us with 4 runs and 512 CTAs).
constexpr long long kRunFixedTiles = 2;
constexpr long long kReduceTiles = 1;

// cluster_cap[n]: clusters of n CTAs the device holds at once (null: every
// grid of one wave, the host rule).
Plan make_plan(int batch, int hkv, int max_seq_len, int chunk, int tile_tokens, int resident, bool merge,
               const int* cluster_cap = nullptr) {
    Plan pl;
    pl.unit_tokens = chunk < tile_tokens ? chunk : tile_tokens;
    pl.units = ceil_div(max_seq_len, pl.unit_tokens);
    const long long heads = static_cast<long long>(batch) * hkv;
    const long long slots = resident > 0 ? resident : 1;
    long long cap = tq::kMaxDecodeCtas / heads;
    if (cap > pl.units) cap = pl.units;
    if (cap < 1) cap = 1;
    auto mergeable = [&](long long n, long long waves) {
        if (!merge) return false;
        if (n == 1) return true;
        if (n > tq::kMaxClusterRuns) return false;
        return cluster_cap != nullptr ? heads <= cluster_cap[n] : waves == 1;
    };
    long long best = 1, best_cost = -1;
    bool best_merged = false;
    auto consider = [&](long long ns) {
        if (ns > cap) ns = cap;
        if (ns < 1) ns = 1;
        const long long run_units = (pl.units + ns - 1) / ns;
        const long long n = (pl.units + run_units - 1) / run_units;  // fewest runs this long
        const long long waves = (heads * n + slots - 1) / slots;
        long long cost = waves * (run_units * pl.unit_tokens + kRunFixedTiles * tile_tokens);
        const bool merged = mergeable(n, waves);
        if (!merged) cost += kReduceTiles * tile_tokens;
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && n < best)) {
            best_cost = cost;
            best = n;
            best_merged = merged;
        }
        return ns;
    };
    for (long long w = (heads + slots - 1) / slots;; ++w)
        if (consider(w * slots / heads) >= cap) break;
    if (merge)
        for (long long n = 1; n <= tq::kMaxClusterRuns; ++n) consider(n);
    pl.n_splits = static_cast<int>(best);
    pl.merged = best_merged;
    pl.waves = (heads * best + slots - 1) / slots;
    return pl;
}

// Fixed runs of `cps` whole chunks (the pages' per-chunk states when cps = 1).
Plan chunk_plan(int max_seq_len, int chunk, int cps) {
    Plan pl;
    pl.unit_tokens = cps * chunk;
    pl.units = ceil_div(max_seq_len, pl.unit_tokens);
    pl.n_splits = pl.units;
    return pl;
}

tq_status device_plan(const Store* cache, int max_seq_len, int chunk, tq_impl impl, Plan* pl,
                      bool merge = true) {
    DeviceFacts* f = nullptr;
    tq_status s = device_facts(&f);
    if (s != TQ_OK) return s;
    const int di = dim_index(cache->head_dim);
    const bool simt = impl == TQ_IMPL_SIMT;
    const int per_sm = simt ? f->simt_ctas[di] : f->mma_ctas[cache->bits == 8 ? 1 : 0][di];
    const int tile = simt ? tq::kSimtTileTokens : tq::mma_tile_tokens(cache->head_dim, cache->bits, false);
    if (cache->paged && chunk < tile) chunk = tile;  // runs start on tile (hence page-aligned) boundaries
    *pl = make_plan(cache->batch, cache->num_kv_heads, max_seq_len, chunk, tile, f->sms * per_sm, merge && !simt,
                    f->clusters[cache->bits == 8 ? 1 : 0][di][cache->paged ? 1 : 0]);
    pl->tile_tokens = tile;
    pl->resident = static_cast<long long>(f->sms) * per_sm;
    // The one-CTA-per-SM layout, for a plan of one wave that either covers
    // at least 95 % of the SMs (each SM's work the same as with three CTAs per
    // SM, without their staggered finish), or has one run per (sequence, kv
    // head) and so no merge at all, or covers at least 75 % with runs of at
    // most 12 stages (the ramp of its ring then dominates: fewer,
    // longer streams fill sooner).  Measured (steps of 20, Llama-70B heads):
    // 1 x 128K 31.5 us (three CTAs per SM: 32.7), 1 x 64K 20.3 (21.1),
    // 1 x 16K 12.0 (12.5), 8 x 8K 22.0 (23.0), 16 x 8K 33.8 (38.1); with
    // longer runs over 84 % of the SMs it lost: 4 x 32K 34.9 (33.2), 8 x 32K
    // 61.5 (58.5).  Grids of several waves keep three CTAs per SM.
    if (!simt && f->wide_ctas > 0 && tq::mma_wide_supported(cache->head_dim, cache->bits, cache->paged)) {
        const int wtile = tq::mma_tile_tokens(cache->head_dim, cache->bits, true);
        const long long wres = static_cast<long long>(f->sms) * f->wide_ctas;
        const Plan w = make_plan(cache->batch, cache->num_kv_heads, max_seq_len, chunk, wtile, static_cast<int>(wres),
                                 merge, f->wide_clusters);
        const long long ctas = static_cast<long long>(w.n_splits) * cache->num_kv_heads * cache->batch;
        const long long run = static_cast<long long>(ceil_div(w.units, w.n_splits)) * w.unit_tokens;
        const bool full = ctas * 20 >= wres * 19;
        const bool no_merge = w.n_splits == 1;
        const bool short_runs = ctas * 4 >= wres * 3 && run <= 12LL * wtile;
        if (w.waves == 1 && (full || no_merge || short_runs)) {
            *pl = w;
            pl->tile_tokens = wtile;
            pl->resident = wres;
            pl->wide = true;
        }
    }
    return TQ_OK;
}

tq_status check_decode_args(const Store* cache, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                            int32_t max_seq_len, int32_t chunk, const void* out) {
    if (q == nullptr || seq_lens == nullptr || out == nullptr) return TQ_ERR_NULL;
    if (!aligned16(q)) return TQ_ERR_ALIGN;
    if (hq < 1 || hq % cache->num_kv_heads != 0) return TQ_ERR_SHAPE;
    if (hq / cache->num_kv_heads > 8) return TQ_ERR_UNSUPPORTED;
    if (max_seq_len < 1) return TQ_ERR_SHAPE;
    if (max_seq_len > cache->capacity) return TQ_ERR_CAPACITY;
    if (chunk < 16 || chunk % 16 != 0) return TQ_ERR_SHAPE;
    return TQ_OK;
}

tq_status run_phase1(const Store* cache, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                     int32_t max_seq_len, float attn_scale, const Plan& pl, float* pm, float* plv, float* pa,
                     int32_t* status, tq_impl impl, cudaStream_t stream, const int32_t* dep_write_pos = nullptr,
                     int32_t dep_n_new = 0, const tq::AppendParams* fused_append = nullptr, bool rotate_q = false,
                     int2* order_buf = nullptr, uint16_t* direct_out = nullptr) {
    if (pl.n_splits > 65535 || cache->num_kv_heads > 65535 || cache->batch > 65535) return TQ_ERR_SHAPE;
    tq::DecodeParams p{};
    p.q = q;
    p.seq_lens = seq_lens;
    p.k_scale = cache->k_scale;
    p.k_bias = cache->k_bias;
    p.v_scale = cache->v_scale;
    p.v_bias = cache->v_bias;
    p.k_codes = cache->k_codes;
    p.v_codes = cache->v_codes;
    p.part_m = pm;
    p.part_l = plv;
    p.part_acc = pa;
    p.status = status;
    p.batch = cache->batch;
    p.num_q_heads = hq;
    p.num_kv_heads = cache->num_kv_heads;
    p.group_q = hq / cache->num_kv_heads;
    p.capacity = cache->capacity;
    p.max_seq_len = max_seq_len;
    p.unit_tokens = pl.unit_tokens;
    p.units = pl.units;
    p.n_splits = pl.n_splits;
    p.score_scale_log2 = attn_scale * 1.4426950408889634f;
    p.dep_write_pos = dep_write_pos;
    p.dep_n_new = dep_n_new;
    p.map = cache->map;
    p.bits = cache->bits;
    p.rotate_q = rotate_q ? 1 : 0;
    p.rot_scale = tq::rotation_scale(cache->head_dim);
    p.app = {};
    if (fused_append != nullptr) {
        if (impl == TQ_IMPL_SIMT) return TQ_ERR_UNSUPPORTED;
        p.app = *fused_append;
    }
    if (impl == TQ_IMPL_SIMT) {
        if (rotate_q) return TQ_ERR_UNSUPPORTED;  // its callers rotate the query first
        // the CUDA-core comparison path reads contiguous int4 caches
        if (cache->paged || cache->bits != 4) return TQ_ERR_UNSUPPORTED;
        return cuda_status(tq::launch_decode_simt(p, cache->head_dim, stream));
    }
    CUtensorMap tm_k, tm_v;
    const int tile = tq::mma_tile_tokens(cache->head_dim, cache->bits, pl.wide);
    p.wide = pl.wide ? 1 : 0;
    tq_status s = make_code_map(&tm_k, cache->k_codes, cache, tile);
    if (s != TQ_OK) return s;
    s = make_code_map(&tm_v, cache->v_codes, cache, tile);
    if (s != TQ_OK) return s;
    // Phase 1 is always a programmatic dependent of the previous kernel on the
    // stream (typically the last step's reduce, which lets its dependents
    // launch once it has seen phase 1 complete), so that its launch overlaps
    // that kernel.  Without an append before it, it waits for that kernel
    // before any read; after an append it waits only before the tiles that
    // hold the new rows.
    p.wait_at_start = dep_write_pos != nullptr ? tq::kWaitForAppend : tq::kWaitAtStart;
    p.out = direct_out;
    // A batch whose grid spans several waves is dispatched longest run first
    // (the lengths are on the device: a one-CTA kernel writes the order).
    const long long ctas = static_cast<long long>(pl.n_splits) * cache->num_kv_heads * cache->batch;
    if (order_buf != nullptr && cache->batch > 1 && pl.resident > 0 && ctas > pl.resident &&
        dep_write_pos == nullptr) {
        tq::OrderParams op{};
        op.seq_lens = seq_lens;
        op.order = order_buf;
        op.status = status;
        op.batch = cache->batch;
        op.max_seq_len = max_seq_len;
        op.units = pl.units;
        op.n_splits = pl.n_splits;
        op.unit_tokens = pl.unit_tokens;
        op.tile_tokens = pl.tile_tokens;
        s = cuda_status(tq::launch_order_runs(op, stream));
        if (s != TQ_OK) return s;
        p.order = order_buf;
    }
    return cuda_status(tq::launch_decode_mma(p, cache->head_dim, tm_k, tm_v, stream, true));
}

}  // namespace

namespace tq {

// Phase 1 + phase 2 with the partial states placed in `partials`
// (`partials_bytes` long, 256-byte aligned) instead of a caller workspace.
// Requests whose partial states do not fit are refused with TQ_ERR_WORKSPACE
// before anything is launched.
tq_status decode_into_partials(const tq_kv_cache* raw, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                               int32_t max_seq_len, float attn_scale, int32_t chunk, uint8_t* partials,
                               size_t partials_bytes, uint16_t* out, int32_t* status, cudaStream_t stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    const Store* cache = &st;
    s = check_decode_args(cache, q, hq, seq_lens, max_seq_len, chunk, out);
    if (s != TQ_OK) return s;
    if (partials == nullptr) return TQ_ERR_WORKSPACE;
    Plan pl;
    s = device_plan(cache, max_seq_len, chunk, TQ_IMPL_MMA, &pl);
    if (s != TQ_OK) return s;
    if (pl.n_splits > kMaxReduceParts) return TQ_ERR_SHAPE;
    const size_t parts = static_cast<size_t>(cache->batch) * hq * pl.n_splits;
    const size_t need = 2 * align256(parts * sizeof(float)) + parts * cache->head_dim * sizeof(float);
    if (need > partials_bytes) return TQ_ERR_WORKSPACE;
    float* pm = reinterpret_cast<float*>(partials);
    float* plv = reinterpret_cast<float*>(partials + align256(parts * sizeof(float)));
    float* pa = reinterpret_cast<float*>(partials + 2 * align256(parts * sizeof(float)));
    if (pl.merged) {  // phase 1 writes the output (one run, or clusters); else as below
        s = run_phase1(cache, q, hq, seq_lens, max_seq_len, attn_scale, pl, pm, plv, pa, status, TQ_IMPL_MMA,
                       stream, nullptr, 0, nullptr, false, nullptr, out);
        if (s == TQ_OK || pl.n_splits == 1) return s;
        cudaGetLastError();  // a refused cluster launch: the partial states and the reduce
    }
    s = run_phase1(cache, q, hq, seq_lens, max_seq_len, attn_scale, pl, pm, plv, pa, status, TQ_IMPL_MMA, stream);
    if (s != TQ_OK) return s;
    ReduceParams r{};
    r.part_m = pm;
    r.part_l = plv;
    r.part_acc = pa;
    r.out = out;
    r.batch = cache->batch;
    r.num_q_heads = hq;
    r.head_dim = cache->head_dim;
    r.n_parts = pl.n_splits;
    return cuda_status(launch_reduce(r, stream, true));
}

tq_status record_cuda_status(cudaError_t e) { return cuda_status(e); }

}  // namespace tq

extern "C" {

int32_t tq_abi_version(void) { return TQ_ABI_VERSION; }

const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_NULL: return "null pointer";
        case TQ_ERR_SHAPE: return "invalid shape";
        case TQ_ERR_CAPACITY: return "exceeds cache capacity";
        case TQ_ERR_WORKSPACE: return "workspace missing or too small";
        case TQ_ERR_CUDA: return "CUDA error";
        case TQ_ERR_UNSUPPORTED: return "unsupported configuration";
        case TQ_ERR_ALIGN: return "misaligned array";
    }
    return "unknown status";
}

int32_t tq_last_cuda_error(void) { return g_last_cuda_error; }

tq_status tq_wait_timeout_selftest(const void* src, int32_t* status, uint32_t limit_us, uint32_t* copied,
                                   void* stream) {
    if (src == nullptr || status == nullptr || copied == nullptr) return TQ_ERR_NULL;
    if (!aligned16(src)) return TQ_ERR_ALIGN;
    if (limit_us < 1 || limit_us > 100000) return TQ_ERR_SHAPE;
    return cuda_status(tq::launch_wait_timeout_selftest(src, status, static_cast<uint64_t>(limit_us) * 1000ull,
                                                        copied, static_cast<cudaStream_t>(stream)));
}

size_t tq_kv_cache_bytes_ex(int32_t batch, int32_t hkv, int32_t head_dim, int32_t group_size, int32_t bits,
                            int32_t capacity) {
    if (batch < 1 || hkv < 1 || capacity < 1 || head_dim < 2 || head_dim % 2 != 0 || group_size < 1 ||
        head_dim % group_size != 0 || (bits != 4 && bits != 8))
        return 0;
    const size_t rows = static_cast<size_t>(batch) * hkv * capacity;
    const size_t codes = align256(rows * (static_cast<size_t>(head_dim) * bits / 8));
    const size_t sb = align256(rows * (head_dim / group_size) * 2);
    return 2 * codes + 4 * sb;
}

size_t tq_kv_cache_bytes(int32_t batch, int32_t hkv, int32_t head_dim, int32_t group_size, int32_t capacity) {
    return tq_kv_cache_bytes_ex(batch, hkv, head_dim, group_size, 4, capacity);
}

tq_status tq_kv_cache_carve_ex(tq_kv_cache* cache, void* base, int32_t batch, int32_t hkv, int32_t head_dim,
                               int32_t group_size, int32_t bits, int32_t capacity) {
    if (cache == nullptr || base == nullptr) return TQ_ERR_NULL;
    if (tq_kv_cache_bytes_ex(batch, hkv, head_dim, group_size, bits, capacity) == 0) return TQ_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(base) & 255u) != 0) return TQ_ERR_ALIGN;
    const size_t rows = static_cast<size_t>(batch) * hkv * capacity;
    const size_t codes = align256(rows * (static_cast<size_t>(head_dim) * bits / 8));
    const size_t sb = align256(rows * (head_dim / group_size) * 2);
    uint8_t* p = static_cast<uint8_t*>(base);
    cache->k_codes = p;
    cache->v_codes = p + codes;
    cache->k_scale = reinterpret_cast<uint16_t*>(p + 2 * codes);
    cache->k_bias = reinterpret_cast<uint16_t*>(p + 2 * codes + sb);
    cache->v_scale = reinterpret_cast<uint16_t*>(p + 2 * codes + 2 * sb);
    cache->v_bias = reinterpret_cast<uint16_t*>(p + 2 * codes + 3 * sb);
    cache->batch = batch;
    cache->num_kv_heads = hkv;
    cache->head_dim = head_dim;
    cache->group_size = group_size;
    cache->capacity = capacity;
    cache->bits = bits;
    return TQ_OK;
}

tq_status tq_kv_cache_carve(tq_kv_cache* cache, void* base, int32_t batch, int32_t hkv, int32_t head_dim,
                            int32_t group_size, int32_t capacity) {
    return tq_kv_cache_carve_ex(cache, base, batch, hkv, head_dim, group_size, 4, capacity);
}

}  // extern "C"

namespace {

tq_status check_append_args(const Store* cache, const uint16_t* k_new, const uint16_t* v_new, int32_t n_new,
                            const int32_t* write_pos) {
    if (k_new == nullptr || v_new == nullptr || write_pos == nullptr) return TQ_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new)) return TQ_ERR_ALIGN;
    if (n_new < 0) return TQ_ERR_SHAPE;
    if (n_new > cache->capacity) return TQ_ERR_CAPACITY;
    return TQ_OK;
}

tq::AppendParams append_params(const Store* cache, const uint16_t* k_new, const uint16_t* v_new,
                               int32_t n_new, const int32_t* write_pos, int32_t* status, uint32_t flags = 0) {
    tq::AppendParams p{};
    p.flags = flags;
    p.rot_scale = tq::rotation_scale(cache->head_dim);
    p.k_new = k_new;
    p.v_new = v_new;
    p.write_pos = write_pos;
    p.k_codes = cache->k_codes;
    p.v_codes = cache->v_codes;
    p.k_scale = cache->k_scale;
    p.k_bias = cache->k_bias;
    p.v_scale = cache->v_scale;
    p.v_bias = cache->v_bias;
    p.status = status;
    p.batch = cache->batch;
    p.num_kv_heads = cache->num_kv_heads;
    p.head_dim = cache->head_dim;
    p.n_new = n_new;
    p.capacity = cache->capacity;
    p.map = cache->map;
    p.bits = cache->bits;
    p.div_ng = tq::make_fastdiv(cache->head_dim / tq::kGroup);
    p.div_n_new = tq::make_fastdiv(n_new > 0 ? n_new : 1);
    p.div_hkv = tq::make_fastdiv(cache->num_kv_heads);
    return p;
}

bool valid_rotation(uint32_t flags) { return (flags & ~(TQ_ROTATE_K | TQ_ROTATE_V)) == 0; }

// A plain (not step-fused) append: large ones take the persistent TMA kernel.
tq_status run_append(const tq::AppendParams& ap, cudaStream_t st) {
    const long long groups =
        static_cast<long long>(ap.batch) * ap.num_kv_heads * ap.n_new * (ap.head_dim / tq::kGroup);
    if (groups >= tq::kTmaAppendMinGroups && groups < (1LL << 31)) {
        CUtensorMap tm_k, tm_v;
        const int box = tq::kTmaAppendBoxRows;
        tq_status s = make_rows_map(&tm_k, ap.k_new, static_cast<unsigned long long>(groups), box);
        if (s == TQ_OK) s = make_rows_map(&tm_v, ap.v_new, static_cast<unsigned long long>(groups), box);
        if (s != TQ_OK) return s;
        DeviceFacts* f = nullptr;
        s = device_facts(&f);
        if (s != TQ_OK) return s;
        return cuda_status(tq::launch_quantize_append_tma(ap, tm_k, tm_v, f->sms, st));
    }
    return cuda_status(tq::launch_quantize_append(ap, st));
}
bool valid_step_flags(uint32_t flags) { return valid_rotation(flags & ~TQ_STEP_ADVANCE); }

// Decode (optionally preceded by an append of n_new rows) with the workspace
// laid out as [m][l][acc][rotated q][run order]; the one path behind tq_decode_step*,
// tq_sdpa_int4_decode*.
tq_status decode_path(const Store* cache, const uint16_t* k_new, const uint16_t* v_new, int32_t n_new,
                      const int32_t* write_pos, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                      int32_t max_seq_len, float attn_scale, int32_t chunk, uint32_t flags, void* workspace,
                      size_t workspace_bytes, uint16_t* out, int32_t* status, tq_impl impl, cudaStream_t st) {
    tq_status s = check_decode_args(cache, q, hq, seq_lens, max_seq_len, chunk, out);
    if (s != TQ_OK) return s;
    if (n_new != 0) {
        s = check_append_args(cache, k_new, v_new, n_new, write_pos);
        if (s != TQ_OK) return s;
    }
    if (!valid_impl(impl) || !valid_step_flags(flags)) return TQ_ERR_UNSUPPORTED;
    const bool advance = (flags & TQ_STEP_ADVANCE) != 0;
    flags &= ~TQ_STEP_ADVANCE;
    if (advance && (write_pos == nullptr || write_pos == seq_lens)) return TQ_ERR_SHAPE;
    const size_t need =
        tq_sdpa_workspace_bytes(cache->batch, hq, cache->num_kv_heads, cache->head_dim, max_seq_len, chunk);
    if (workspace == nullptr || workspace_bytes < need) return TQ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TQ_ERR_ALIGN;
    Plan pl;
    // the runs may merge in phase 1 unless the reduce has other work (the
    // output rotation of TQ_ROTATE_V, the length advance)
    s = device_plan(cache, max_seq_len, chunk, impl, &pl, !(flags & TQ_ROTATE_V) && !advance);
    if (s != TQ_OK) return s;
    if (pl.n_splits > tq::kMaxReduceParts) return TQ_ERR_SHAPE;
    const size_t parts = static_cast<size_t>(cache->batch) * hq * pl.n_splits;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* pm = reinterpret_cast<float*>(ws);
    float* plv = reinterpret_cast<float*>(ws + align256(parts * sizeof(float)));
    float* pa = reinterpret_cast<float*>(ws + 2 * align256(parts * sizeof(float)));
    uint16_t* q_rot = reinterpret_cast<uint16_t*>(ws + 2 * align256(parts * sizeof(float)) +
                                                  align256(parts * cache->head_dim * sizeof(float)));
    int2* order = reinterpret_cast<int2*>(reinterpret_cast<uint8_t*>(q_rot) +
                                                align256(static_cast<size_t>(cache->batch) * hq *
                                                         cache->head_dim * sizeof(uint16_t)));
    const float rs = tq::rotation_scale(cache->head_dim);
    const tq_impl ph1 = impl == TQ_IMPL_SIMT ? TQ_IMPL_SIMT : TQ_IMPL_MMA;
    // keys stored rotated: attend with the rotated query, (H q).(H k) = q.k;
    // the tensor-core kernel rotates each query head as it loads it
    const bool rotate_q = (flags & TQ_ROTATE_K) != 0 && ph1 == TQ_IMPL_MMA;
    if ((flags & TQ_ROTATE_K) && !rotate_q) {
        s = cuda_status(tq::launch_rotate_rows(q, static_cast<long long>(cache->batch) * hq, cache->head_dim, q_rot,
                                               rs, st));
        if (s != TQ_OK) return s;
        q = q_rot;
    }
    // A few new rows per sequence are quantized (and rotated, for head dims
    // up to 128, whose rows fit one warp) by the decode kernel itself: the CTA
    // that reads them writes them first.  Longer appends, and rotated ones of
    // wider heads, run the append kernel; the decode starts early and waits
    // only for the tiles that hold the new rows.
    const tq::AppendParams ap = append_params(cache, k_new, v_new, n_new, write_pos, status, flags);
    const bool fused = n_new > 0 && n_new <= tq::kFusedAppendMaxRows && ph1 == TQ_IMPL_MMA;
    if (n_new > 0 && !fused) {
        s = cuda_status(tq::launch_quantize_append_primary(ap, st));
        if (s != TQ_OK) return s;
    }
    const bool dep = n_new > 0 && !fused && ph1 == TQ_IMPL_MMA;
    // Phase 1 writes the output itself and no reduce is launched when the plan
    // says so (never when the reduce has other work: the output rotation of
    // TQ_ROTATE_V, the length advance): one run per sequence, or up to
    // kMaxClusterRuns runs whose clusters (one per sequence and kv head, merging
    // their states in shared memory) the device holds all at once.
    const bool direct = ph1 == TQ_IMPL_MMA && !(flags & TQ_ROTATE_V) && !advance && pl.merged;
    bool own_out = direct;
    s = run_phase1(cache, q, hq, seq_lens, max_seq_len, attn_scale, pl, pm, plv, pa, status, ph1, st,
                   dep ? write_pos : nullptr, dep ? n_new : 0, fused ? &ap : nullptr, rotate_q, order,
                   own_out ? out : nullptr);
    if (s != TQ_OK && own_out && pl.n_splits > 1) {
        // a cluster launch the device refused (nothing was queued; e.g. a GPU
        // partition too small to place the cluster): the same runs with
        // partial states and the reduce, the same output
        cudaGetLastError();
        own_out = false;
        s = run_phase1(cache, q, hq, seq_lens, max_seq_len, attn_scale, pl, pm, plv, pa, status, ph1, st,
                       dep ? write_pos : nullptr, dep ? n_new : 0, fused ? &ap : nullptr, rotate_q, order, nullptr);
    }
    if (s != TQ_OK) return s;
    tq::ReduceParams r{};
    r.part_m = pm;
    r.part_l = plv;
    r.part_acc = pa;
    r.out = out;
    r.batch = cache->batch;
    r.num_q_heads = hq;
    r.head_dim = cache->head_dim;
    r.n_parts = pl.n_splits;
    r.rotate_out = (flags & TQ_ROTATE_V) ? 1 : 0;
    r.rot_scale = rs;
    // TQ_STEP_ADVANCE: the reduce advances the lengths once phase 1 is done
    // (which covers a fused append); after a separate append kernel a plain
    // launch after the reduce does it, so that stream order covers that kernel
    if (advance && (fused || n_new == 0)) {
        r.adv_seq_lens = const_cast<int32_t*>(seq_lens);
        r.adv_write_pos = const_cast<int32_t*>(write_pos);
        r.adv_n = n_new;
    }
    if (own_out) return s;
    s = cuda_status(tq::launch_reduce(r, st, true));
    if (s != TQ_OK || !advance || fused || n_new == 0) return s;
    return cuda_status(tq::launch_advance(const_cast<int32_t*>(seq_lens), const_cast<int32_t*>(write_pos),
                                          cache->batch, n_new, st));
}

}  // namespace

extern "C" {

tq_status tq_quantize_kv_append(const tq_kv_cache* cache, const uint16_t* k_new, const uint16_t* v_new,
                                int32_t n_new, const int32_t* write_pos, int32_t* status, void* stream) {
    return tq_quantize_kv_append_ex(cache, k_new, v_new, n_new, write_pos, 0u, status, stream);
}

tq_status tq_decode_step(const tq_kv_cache* cache, const uint16_t* k_new, const uint16_t* v_new, int32_t n_new,
                         const int32_t* write_pos, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                         int32_t max_seq_len, float attn_scale, int32_t chunk, void* workspace,
                         size_t workspace_bytes, uint16_t* out, int32_t* status, void* stream) {
    return tq_decode_step_ex(cache, k_new, v_new, n_new, write_pos, q, hq, seq_lens, max_seq_len, attn_scale, chunk,
                             0u, workspace, workspace_bytes, out, status, stream);
}

tq_status tq_decode_step_ex(const tq_kv_cache* raw, const uint16_t* k_new, const uint16_t* v_new, int32_t n_new,
                            const int32_t* write_pos, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                            int32_t max_seq_len, float attn_scale, int32_t chunk, uint32_t flags, void* workspace,
                            size_t workspace_bytes, uint16_t* out, int32_t* status, void* stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    const Store* cache = &st;
    s = check_append_args(cache, k_new, v_new, n_new, write_pos);
    if (s != TQ_OK) return s;
    return decode_path(cache, k_new, v_new, n_new, write_pos, q, hq, seq_lens, max_seq_len, attn_scale, chunk, flags,
                       workspace, workspace_bytes, out, status, TQ_IMPL_MMA, static_cast<cudaStream_t>(stream));
}

tq_status tq_quantize_kv_append_ex(const tq_kv_cache* raw, const uint16_t* k_new, const uint16_t* v_new,
                                   int32_t n_new, const int32_t* write_pos, uint32_t flags, int32_t* status,
                                   void* stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    const Store* cache = &st;
    s = check_append_args(cache, k_new, v_new, n_new, write_pos);
    if (s != TQ_OK) return s;
    if (!valid_rotation(flags)) return TQ_ERR_UNSUPPORTED;
    if (n_new == 0) return TQ_OK;
    return run_append(append_params(cache, k_new, v_new, n_new, write_pos, status, flags),
                      static_cast<cudaStream_t>(stream));
}

tq_status tq_hadamard_rotate(const uint16_t* x, int64_t rows, int32_t dim, uint16_t* out, void* stream) {
    if (x == nullptr || out == nullptr) return TQ_ERR_NULL;
    if (rows < 0) return TQ_ERR_SHAPE;
    if (!supported_dim(dim)) return TQ_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(out)) return TQ_ERR_ALIGN;
    return cuda_status(tq::launch_rotate_rows(x, rows, dim, out, tq::rotation_scale(dim),
                                              static_cast<cudaStream_t>(stream)));
}

size_t tq_sdpa_workspace_bytes(int32_t batch, int32_t hq, int32_t hkv, int32_t head_dim, int32_t max_seq_len,
                               int32_t chunk) {
    if (batch < 1 || hq < 1 || hkv < 1 || head_dim < 1 || max_seq_len < 1 || chunk < 1) return 0;
    // n_splits <= min(units of the smallest unit (16 or chunk tokens), kMaxDecodeCtas / (batch * hkv))
    const long long unit = chunk < 16 ? chunk : 16;
    long long ns = (max_seq_len + unit - 1) / unit;
    long long cap = tq::kMaxDecodeCtas / (static_cast<long long>(batch) * hkv);
    if (cap < 1) cap = 1;
    if (ns > cap) ns = cap;
    const size_t parts = static_cast<size_t>(batch) * hq * static_cast<size_t>(ns);
    // m, l, acc of every part, the rotated query (TQ_ROTATE_K), the dispatch
    // order of the runs
    return 2 * align256(parts * sizeof(float)) + align256(parts * head_dim * sizeof(float)) +
           align256(static_cast<size_t>(batch) * hq * head_dim * sizeof(uint16_t)) +
           align256(static_cast<size_t>(batch) * static_cast<size_t>(ns) * sizeof(int2));
}

tq_status tq_sdpa_int4_decode_impl(const tq_kv_cache* raw, const uint16_t* q, int32_t hq,
                                   const int32_t* seq_lens, int32_t max_seq_len, float attn_scale, int32_t chunk,
                                   void* workspace, size_t workspace_bytes, uint16_t* out, int32_t* status,
                                   tq_impl impl, void* stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    return decode_path(&st, nullptr, nullptr, 0, nullptr, q, hq, seq_lens, max_seq_len, attn_scale, chunk, 0u,
                       workspace, workspace_bytes, out, status, impl, static_cast<cudaStream_t>(stream));
}

tq_status tq_sdpa_int4_decode_ex(const tq_kv_cache* raw, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                                 int32_t max_seq_len, float attn_scale, int32_t chunk, uint32_t flags,
                                 void* workspace, size_t workspace_bytes, uint16_t* out, int32_t* status,
                                 void* stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    if (!valid_rotation(flags)) return TQ_ERR_UNSUPPORTED;
    return decode_path(&st, nullptr, nullptr, 0, nullptr, q, hq, seq_lens, max_seq_len, attn_scale, chunk, flags,
                       workspace, workspace_bytes, out, status, TQ_IMPL_AUTO, static_cast<cudaStream_t>(stream));
}

size_t tq_host_staging_bytes(int32_t batch, int32_t hq, int32_t hkv, int32_t head_dim, int32_t n_new) {
    if (batch < 1 || hq < 1 || hkv < 1 || head_dim < 1 || n_new < 0) return 0;
    const size_t qb = static_cast<size_t>(batch) * hq * head_dim * 2;
    const size_t kb = static_cast<size_t>(batch) * hkv * n_new * head_dim * 2;
    return 2 * align256(qb) + 2 * align256(kb);  // q, out, k_new, v_new
}

tq_status tq_decode_step_host(const tq_kv_cache* cache, const uint16_t* h_k_new, const uint16_t* h_v_new,
                              int32_t n_new, const int32_t* write_pos, const uint16_t* h_q, int32_t hq,
                              const int32_t* seq_lens, int32_t max_seq_len, float attn_scale, int32_t chunk,
                              uint32_t flags, void* workspace, size_t workspace_bytes, void* staging,
                              size_t staging_bytes, uint16_t* h_out, int32_t* status, void* stream) {
    if (cache == nullptr || h_q == nullptr || h_out == nullptr || staging == nullptr) return TQ_ERR_NULL;
    if (n_new > 0 && (h_k_new == nullptr || h_v_new == nullptr)) return TQ_ERR_NULL;
    if (hq < 1 || n_new < 0) return TQ_ERR_SHAPE;
    const size_t need = tq_host_staging_bytes(cache->batch, hq, cache->num_kv_heads, cache->head_dim, n_new);
    if (need == 0) return TQ_ERR_SHAPE;
    if (staging_bytes < need) return TQ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0) return TQ_ERR_ALIGN;
    // Page-locked host buffers are addressable from the GPU (over NVLink-C2C on
    // Grace-Blackwell): then the step reads q / k_new / v_new and writes the
    // output in place, with no copy-engine round trips.  Other host memory
    // goes through the staging copies.
    auto mapped = [](const void* ptr) -> void* {
        if (ptr == nullptr) return nullptr;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
    };
    {
        void* dq = mapped(h_q);
        void* dout = mapped(h_out);
        void* dk = n_new > 0 ? mapped(h_k_new) : dq;
        void* dv = n_new > 0 ? mapped(h_v_new) : dq;
        if (dq != nullptr && dout != nullptr && dk != nullptr && dv != nullptr && aligned16(dq) && aligned16(dk) &&
            aligned16(dv))
            return tq_decode_step_ex(cache, static_cast<const uint16_t*>(dk), static_cast<const uint16_t*>(dv),
                                     n_new, write_pos, static_cast<const uint16_t*>(dq), hq, seq_lens, max_seq_len,
                                     attn_scale, chunk, flags, workspace, workspace_bytes,
                                     static_cast<uint16_t*>(dout), status, stream);
    }
    const size_t qb = static_cast<size_t>(cache->batch) * hq * cache->head_dim * 2;
    const size_t kb = static_cast<size_t>(cache->batch) * cache->num_kv_heads * n_new * cache->head_dim * 2;
    uint8_t* st = static_cast<uint8_t*>(staging);
    uint16_t* d_q = reinterpret_cast<uint16_t*>(st);
    uint16_t* d_out = reinterpret_cast<uint16_t*>(st + align256(qb));
    uint16_t* d_k = reinterpret_cast<uint16_t*>(st + 2 * align256(qb));
    uint16_t* d_v = reinterpret_cast<uint16_t*>(st + 2 * align256(qb) + align256(kb));
    cudaStream_t s_ = static_cast<cudaStream_t>(stream);
    tq_status s = cuda_status(cudaMemcpyAsync(d_q, h_q, qb, cudaMemcpyHostToDevice, s_));
    if (s == TQ_OK && kb > 0) s = cuda_status(cudaMemcpyAsync(d_k, h_k_new, kb, cudaMemcpyHostToDevice, s_));
    if (s == TQ_OK && kb > 0) s = cuda_status(cudaMemcpyAsync(d_v, h_v_new, kb, cudaMemcpyHostToDevice, s_));
    if (s != TQ_OK) return s;
    s = tq_decode_step_ex(cache, d_k, d_v, n_new, write_pos, d_q, hq, seq_lens, max_seq_len, attn_scale, chunk,
                          flags, workspace, workspace_bytes, d_out, status, stream);
    if (s != TQ_OK) return s;
    return cuda_status(cudaMemcpyAsync(h_out, d_out, qb, cudaMemcpyDeviceToHost, s_));
}

size_t tq_paged_kv_cache_bytes(int32_t num_pages, int32_t hkv, int32_t head_dim, int32_t group_size, int32_t bits,
                               int32_t page_tokens) {
    return tq_kv_cache_bytes_ex(num_pages, hkv, head_dim, group_size, bits, page_tokens);  // a page = one row block
}

tq_status tq_paged_kv_cache_carve(tq_paged_kv_cache* cache, void* base, const int32_t* block_table, int32_t batch,
                                  int32_t hkv, int32_t head_dim, int32_t group_size, int32_t bits,
                                  int32_t page_tokens, int32_t num_pages, int32_t max_pages_per_seq) {
    if (cache == nullptr || base == nullptr || block_table == nullptr) return TQ_ERR_NULL;
    if (batch < 1 || max_pages_per_seq < 1 || page_tokens % kPageTokenMultiple != 0) return TQ_ERR_SHAPE;
    tq_kv_cache pool;
    tq_status s = tq_kv_cache_carve_ex(&pool, base, num_pages, hkv, head_dim, group_size, bits, page_tokens);
    if (s != TQ_OK) return s;
    cache->k_codes = pool.k_codes;
    cache->v_codes = pool.v_codes;
    cache->k_scale = pool.k_scale;
    cache->k_bias = pool.k_bias;
    cache->v_scale = pool.v_scale;
    cache->v_bias = pool.v_bias;
    cache->block_table = block_table;
    cache->batch = batch;
    cache->num_kv_heads = hkv;
    cache->head_dim = head_dim;
    cache->group_size = group_size;
    cache->page_tokens = page_tokens;
    cache->num_pages = num_pages;
    cache->max_pages_per_seq = max_pages_per_seq;
    cache->bits = bits;
    return TQ_OK;
}

tq_status tq_paged_quantize_kv_append(const tq_paged_kv_cache* raw, const uint16_t* k_new, const uint16_t* v_new,
                                      int32_t n_new, const int32_t* write_pos, uint32_t flags, int32_t* status,
                                      void* stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    s = check_append_args(&st, k_new, v_new, n_new, write_pos);
    if (s != TQ_OK) return s;
    if (!valid_rotation(flags)) return TQ_ERR_UNSUPPORTED;
    if (n_new == 0) return TQ_OK;
    return run_append(append_params(&st, k_new, v_new, n_new, write_pos, status, flags),
                      static_cast<cudaStream_t>(stream));
}

tq_status tq_paged_sdpa_int4_decode(const tq_paged_kv_cache* raw, const uint16_t* q, int32_t hq,
                                    const int32_t* seq_lens, int32_t max_seq_len, float attn_scale, int32_t chunk,
                                    uint32_t flags, void* workspace, size_t workspace_bytes, uint16_t* out,
                                    int32_t* status, void* stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    if (!valid_rotation(flags)) return TQ_ERR_UNSUPPORTED;
    return decode_path(&st, nullptr, nullptr, 0, nullptr, q, hq, seq_lens, max_seq_len, attn_scale, chunk, flags,
                       workspace, workspace_bytes, out, status, TQ_IMPL_MMA, static_cast<cudaStream_t>(stream));
}

tq_status tq_paged_decode_step(const tq_paged_kv_cache* raw, const uint16_t* k_new, const uint16_t* v_new,
                               int32_t n_new, const int32_t* write_pos, const uint16_t* q, int32_t hq,
                               const int32_t* seq_lens, int32_t max_seq_len, float attn_scale, int32_t chunk,
                               uint32_t flags, void* workspace, size_t workspace_bytes, uint16_t* out,
                               int32_t* status, void* stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    s = check_append_args(&st, k_new, v_new, n_new, write_pos);
    if (s != TQ_OK) return s;
    return decode_path(&st, k_new, v_new, n_new, write_pos, q, hq, seq_lens, max_seq_len, attn_scale, chunk, flags,
                       workspace, workspace_bytes, out, status, TQ_IMPL_MMA, static_cast<cudaStream_t>(stream));
}

tq_status tq_sdpa_int4_decode(const tq_kv_cache* cache, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                              int32_t max_seq_len, float attn_scale, int32_t chunk, void* workspace,
                              size_t workspace_bytes, uint16_t* out, int32_t* status, void* stream) {
    return tq_sdpa_int4_decode_impl(cache, q, hq, seq_lens, max_seq_len, attn_scale, chunk, workspace,
                                    workspace_bytes, out, status, TQ_IMPL_AUTO, stream);
}

tq_status tq_sdpa_plan(const tq_kv_cache* cache, int32_t hq, int32_t max_seq_len, int32_t chunk, tq_impl impl,
                       int32_t* n_splits, int32_t* max_run_tokens) {
    if (cache == nullptr || n_splits == nullptr || max_run_tokens == nullptr) return TQ_ERR_NULL;
    if (!supported_dim(cache->head_dim)) return TQ_ERR_UNSUPPORTED;
    if (cache->batch < 1 || cache->num_kv_heads < 1 || hq < 1 || max_seq_len < 1 || chunk < 16 || chunk % 16)
        return TQ_ERR_SHAPE;
    if (!valid_impl(impl)) return TQ_ERR_UNSUPPORTED;
    Plan pl;
    const Store st = shape_of(cache);
    tq_status s = device_plan(&st, max_seq_len, chunk, impl, &pl);
    if (s != TQ_OK) return s;
    *n_splits = pl.n_splits;
    *max_run_tokens = ceil_div(pl.units, pl.n_splits) * pl.unit_tokens;
    return TQ_OK;
}

tq_status tq_split_plan(int32_t batch, int32_t num_kv_heads, int32_t max_seq_len, int32_t chunk,
                        int32_t tile_tokens, int32_t resident_ctas, int32_t merge, int32_t* n_splits,
                        int32_t* max_run_tokens) {
    if (n_splits == nullptr || max_run_tokens == nullptr) return TQ_ERR_NULL;
    if (batch < 1 || num_kv_heads < 1 || max_seq_len < 1 || chunk < 16 || chunk % 16 || tile_tokens < 16 ||
        tile_tokens % 16 || resident_ctas < 1)
        return TQ_ERR_SHAPE;
    const Plan pl = make_plan(batch, num_kv_heads, max_seq_len, chunk, tile_tokens, resident_ctas, merge != 0);
    *n_splits = pl.n_splits;
    *max_run_tokens = ceil_div(pl.units, pl.n_splits) * pl.unit_tokens;
    return TQ_OK;
}

tq_status tq_sdpa_int4_partial(const tq_kv_cache* raw, const uint16_t* q, int32_t hq, const int32_t* seq_lens,
                               int32_t max_seq_len, float attn_scale, int32_t chunk, int32_t chunks_per_split,
                               float* part_m, float* part_l, float* part_acc, int32_t* status, tq_impl impl,
                               void* stream) {
    Store st;
    tq_status s = store_of(raw, &st);
    if (s != TQ_OK) return s;
    const Store* cache = &st;
    s = check_decode_args(cache, q, hq, seq_lens, max_seq_len, chunk, part_m);
    if (s != TQ_OK) return s;
    if (part_l == nullptr || part_acc == nullptr) return TQ_ERR_NULL;
    if (!valid_impl(impl)) return TQ_ERR_UNSUPPORTED;
    if (chunks_per_split < 0) return TQ_ERR_SHAPE;
    Plan pl;
    if (chunks_per_split == 0) {
        s = device_plan(cache, max_seq_len, chunk, impl, &pl);
        if (s != TQ_OK) return s;
    } else {
        pl = chunk_plan(max_seq_len, chunk, chunks_per_split);
    }
    return run_phase1(cache, q, hq, seq_lens, max_seq_len, attn_scale, pl, part_m, part_l, part_acc, status,
                      impl == TQ_IMPL_SIMT ? TQ_IMPL_SIMT : TQ_IMPL_MMA, static_cast<cudaStream_t>(stream));
}

tq_status tq_sdpa_int4_reduce(const float* part_m, const float* part_l, const float* part_acc, int32_t batch,
                              int32_t hq, int32_t head_dim, int32_t n_parts, uint16_t* out, void* stream) {
    if (part_m == nullptr || part_l == nullptr || part_acc == nullptr || out == nullptr) return TQ_ERR_NULL;
    if (batch < 1 || hq < 1 || head_dim < 1 || n_parts < 1 || n_parts > tq::kMaxReduceParts) return TQ_ERR_SHAPE;
    if (!supported_dim(head_dim)) return TQ_ERR_UNSUPPORTED;
    tq::ReduceParams r{};
    r.part_m = part_m;
    r.part_l = part_l;
    r.part_acc = part_acc;
    r.out = out;
    r.batch = batch;
    r.num_q_heads = hq;
    r.head_dim = head_dim;
    r.n_parts = n_parts;
    return cuda_status(tq::launch_reduce(r, static_cast<cudaStream_t>(stream), false));
}

tq_status tq_dequantize_kv(const tq_kv_cache* cache, int32_t n_rows, uint16_t* k_out, uint16_t* v_out,
                           void* stream) {
    tq_status s = check_cache(cache);
    if (s != TQ_OK) return s;
    if (k_out == nullptr || v_out == nullptr) return TQ_ERR_NULL;
    if (n_rows < 0) return TQ_ERR_SHAPE;
    if (n_rows > cache->capacity) return TQ_ERR_CAPACITY;
    if (!aligned16(k_out) || !aligned16(v_out)) return TQ_ERR_ALIGN;
    if (n_rows == 0) return TQ_OK;
    DeviceFacts* f = nullptr;
    s = device_facts(&f);
    if (s != TQ_OK) return s;
    tq::DequantParams p{};
    p.k_codes = cache->k_codes;
    p.v_codes = cache->v_codes;
    p.k_scale = cache->k_scale;
    p.k_bias = cache->k_bias;
    p.v_scale = cache->v_scale;
    p.v_bias = cache->v_bias;
    p.k_out = k_out;
    p.v_out = v_out;
    p.batch = cache->batch;
    p.num_kv_heads = cache->num_kv_heads;
    p.head_dim = cache->head_dim;
    p.capacity = cache->capacity;
    p.n_rows = n_rows;
    p.bits = cache->bits;
    return cuda_status(tq::launch_dequant(p, f->sms, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

/*
 * tq.h -- C ABI of the int4 KV-cache decode path for NVIDIA GB300 (sm_103a).
 *
 * Two operations, as the pages describe the method:
 *
 *   quantize-on-store   fp16 K/V rows -> packed int4 codes + fp16 scale/bias,
 *                       written in place into a preallocated cache
 *                       ("turboquant-llama3.170B" README, decode-step listing:
 *                        RoPE, then quantize K,V to int4, then fused sdpa_int4;
 *                        "Fused int4 Attention for Gemma 4 31B", Background:
 *                        MLX-style int4 with a per-group scale and bias).
 *   fused decode attention (sdpa_int4)
 *                       one query token per sequence attends over the int4
 *                       cache; dequantisation happens in registers, softmax is
 *                       online, the sequence is split into chunks (512 tokens by
 *                       default) whose partial softmax states are merged by a
 *                       log-sum-exp reduce ("turboquant-llama3.170B" README,
 *                       kernel paragraph and split-K paragraph; Gemma page,
 *                       "What I Built Instead": sdpa_int4(Q, K_int4, V_int4)).
 *
 * Conventions shared by every entry point
 *   - All array pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory and keeps no per-call state between calls.
 *   - fp16 values are passed as uint16_t holding IEEE binary16 bits.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and never synchronise the host.
 *   - Host-side argument checks run before any launch and return a status;
 *     nothing is launched when a check fails.  TQ_ERR_CUDA means a launch was
 *     attempted and CUDA reported an error; tq_last_cuda_error() returns it.
 *   - Kernels never trap.  Device-detected problems (a write position past the
 *     cache capacity, a length outside [0, max_seq_len], a pipeline wait that
 *     timed out) skip the offending work and OR a TQ_DEV_* bit into the
 *     optional `status` word (device int32, may be NULL).  The caller zeroes it
 *     when it wants to start afresh.
 *   - Inputs containing NaN or Inf give unspecified (but finite-time) results.
 *
 * Cache layout (one cache = one attention layer), all row-major:
 *   k_codes, v_codes  uint8  [batch][num_kv_heads][capacity][head_dim / 2]
 *                     element 2i of a row is the low nibble of byte i
 *                     (the Gemma page reads codes with masks 0xF, 0xF0, ...,
 *                      low nibble first)
 *   k_scale, k_bias,  fp16   [batch][num_kv_heads][capacity][head_dim / 64]
 *   v_scale, v_bias          one (scale, bias) per group of 64 consecutive
 *                            head_dim elements; value ~ scale * code + bias
 * Requirements: head_dim in {64, 128, 256}; group_size == 64; capacity a
 * positive multiple of 16; every array 16-byte aligned (256 recommended).
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_ABI_VERSION 2
#define TQ_GROUP_SIZE 64
#define TQ_DEFAULT_CHUNK 512

typedef enum tq_status {
    TQ_OK = 0,
    TQ_ERR_NULL = 1,        /* a required pointer is NULL */
    TQ_ERR_SHAPE = 2,       /* inconsistent or out-of-range sizes */
    TQ_ERR_CAPACITY = 3,    /* max_seq_len (or n_new) larger than the cache capacity */
    TQ_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than required */
    TQ_ERR_CUDA = 5,        /* CUDA reported an error (see tq_last_cuda_error) */
    TQ_ERR_UNSUPPORTED = 6, /* head_dim / group / GQA ratio / impl not implemented */
    TQ_ERR_ALIGN = 7        /* an array is not 16-byte (workspace: 256-byte) aligned */
} tq_status;

/* Bits ORed into the optional device status word. */
#define TQ_DEV_WRITE_POS 0x1 /* append: write_pos[b] < 0 or write_pos[b] + n_new > capacity; rows skipped */
#define TQ_DEV_SEQ_LEN 0x2   /* decode: seq_lens[b] < 0 or > max_seq_len; clamped into range */
#define TQ_DEV_TIMEOUT 0x4   /* a pipeline wait exceeded its time limit; the CTA gave up */
#define TQ_DEV_PAGE 0x8      /* paged cache: a block-table entry outside [0, num_pages); page 0 used instead */

/* Rotation flags ("Running and Evaluating TurboQuant optimized Gemma 4",
 * TurboQuant section: vectors are rotated by the normalised Sylvester Hadamard
 * matrix H = H_n / sqrt(n) before quantisation, which spreads outliers over
 * all coordinates; H is its own inverse).  In this library H is applied by an
 * fp32 fast transform (stages h = 1, 2, ..., n/2) and rounded to fp16.
 *   TQ_ROTATE_K  keys are stored as quantize(H k); decode then uses H q, and
 *                (H q).(H k) = q.k leaves the scores unchanged.
 *   TQ_ROTATE_V  values are stored as quantize(H v); decode returns H o of the
 *                attention output o over them, which is the output over v. */
#define TQ_ROTATE_K 0x1u
#define TQ_ROTATE_V 0x2u

/* tq_decode_step_ex / tq_paged_decode_step: after the step, add n_new to
 * write_pos[b] and to seq_lens[b] on the device (both arrays are written;
 * they must not overlap).  A step captured once in a CUDA graph can then be
 * replayed token after token with no host work; the graph keeps the
 * max_seq_len it was captured with, which must stay an upper bound of the
 * advancing lengths. */
#define TQ_STEP_ADVANCE 0x100u

/* Decode implementations (tq_sdpa_int4_decode_impl and friends). */
typedef enum tq_impl {
    TQ_IMPL_AUTO = 0, /* the tensor-core path */
    TQ_IMPL_MMA = 1,  /* mma.sync tensor-core tiles fed by TMA */
    TQ_IMPL_SIMT = 2  /* CUDA-core fp32 path (comparison baseline) */
} tq_impl;

typedef struct tq_kv_cache {
    uint8_t* k_codes;  /* [B][Hkv][cap][D * bits / 8] */
    uint8_t* v_codes;  /* [B][Hkv][cap][D * bits / 8] */
    uint16_t* k_scale; /* [B][Hkv][cap][D/64] fp16 */
    uint16_t* k_bias;
    uint16_t* v_scale;
    uint16_t* v_bias;
    int32_t batch;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t group_size; /* must be 64 */
    int32_t capacity;   /* tokens per (sequence, kv head) */
    int32_t bits;       /* code width: 4 (two codes per byte, element 2i in the low
                           nibble of byte i) or 8 (one code per byte; the
                           TurboQuant Gemma 4 page's --kv-bits 8), every
                           head_dim */
} tq_kv_cache;

/* Paged cache: a pool of pages, each holding page_tokens consecutive tokens of
 * one sequence for every kv head, and a block table mapping each sequence's
 * logical pages to pool pages (for ragged batches: the "turboquant-llama3.170B"
 * README's 18% concatenation gap is what a cache that grows by reallocation
 * costs).  Row t of (sequence b, kv head h) is row
 * t % page_tokens of head h in page block_table[b * max_pages_per_seq +
 * t / page_tokens].  The caller owns the pool and the table and allocates
 * pages before appending into them; a table entry outside [0, num_pages) sets
 * TQ_DEV_PAGE and page 0 is used instead (no fault). */
typedef struct tq_paged_kv_cache {
    uint8_t* k_codes;  /* [num_pages][Hkv][page_tokens][D * bits / 8] */
    uint8_t* v_codes;
    uint16_t* k_scale; /* [num_pages][Hkv][page_tokens][D/64] fp16 */
    uint16_t* k_bias;
    uint16_t* v_scale;
    uint16_t* v_bias;
    const int32_t* block_table; /* device [batch][max_pages_per_seq] */
    int32_t batch;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t group_size;  /* must be 64 */
    int32_t page_tokens; /* a multiple of 128 */
    int32_t num_pages;
    int32_t max_pages_per_seq; /* logical capacity = max_pages_per_seq * page_tokens */
    int32_t bits;              /* code width, as in tq_kv_cache */
} tq_paged_kv_cache;

/* ABI version of the loaded library (TQ_ABI_VERSION it was built with). */
int32_t tq_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* tq_status_string(tq_status s);

/* The cudaError_t of the most recent TQ_ERR_CUDA on the calling host thread. */
int32_t tq_last_cuda_error(void);

/* Diagnostic of the device-side failure path (no counterpart on the pages):
 * the decode kernels wait on their pipeline stages with a time limit and,
 * when a wait runs out, OR TQ_DEV_TIMEOUT into the status word and leave.
 * This call runs that wait on one CTA: it copies 1,024 bytes from `src`
 * (device, 16-byte aligned) into shared memory and waits for the copy, then
 * waits on a barrier that nothing arrives at, giving up after `limit_us`
 * microseconds (1..100000).  It then ORs TQ_DEV_TIMEOUT into *status and
 * writes to *copied the sum (mod 2^32) of the 256 32-bit words it copied
 * (0xFFFFFFFF if even the copy had not landed).  Nothing is in flight when
 * the kernel ends.  Null pointers: TQ_ERR_NULL; misaligned src:
 * TQ_ERR_ALIGN; limit out of range: TQ_ERR_SHAPE. */
tq_status tq_wait_timeout_selftest(const void* src, int32_t* status, uint32_t limit_us,
                                   uint32_t* copied, void* stream);

/* Bytes of the six cache arrays together, each rounded up to 256 bytes, as
 * laid out by tq_kv_cache_carve.  0 for invalid sizes.  Host-only. */
size_t tq_kv_cache_bytes(int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                         int32_t group_size, int32_t capacity);

/* Point the six arrays of *cache into one caller-owned allocation `base` of
 * at least tq_kv_cache_bytes(...) bytes (256-byte aligned), and fill in the
 * sizes.  Order: k_codes, v_codes, k_scale, k_bias, v_scale, v_bias.
 * Host-only (no device access). */
tq_status tq_kv_cache_carve(tq_kv_cache* cache, void* base, int32_t batch,
                            int32_t num_kv_heads, int32_t head_dim,
                            int32_t group_size, int32_t capacity);

/* The same for a code width of `bits` (4 or 8); the two functions above are
 * bits = 4 (and tq_kv_cache_carve sets cache->bits = 4). */
size_t tq_kv_cache_bytes_ex(int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                            int32_t group_size, int32_t bits, int32_t capacity);
tq_status tq_kv_cache_carve_ex(tq_kv_cache* cache, void* base, int32_t batch,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t group_size, int32_t bits, int32_t capacity);

/* Quantize-on-store.
 * k_new, v_new: fp16 [batch][num_kv_heads][n_new][head_dim], contiguous.
 * write_pos:    device int32 [batch]; token i of sequence b goes to cache row
 *               write_pos[b] + i.  The caller advances its lengths afterwards.
 * Per group of 64 elements x_0..x_63 (fp32 arithmetic, round-to-nearest-even):
 *   mn, mx = min, max;  scale = fp16(fp32(mx - mn) / 15);  bias = fp16(mn)
 *   code_i = clamp(rint(fp32(x_i - bias) / float(scale)), 0, 15), or 0 when
 *   float(scale) == 0;  a zero minimum is stored as +0, and mx is the first
 *   element holding the largest value (so a group of zeros opening with -0
 *   stores scale -0).
 * Bit-identical to the CPU oracle.  Rows with an out-of-range write position
 * are skipped and TQ_DEV_WRITE_POS is set. */
tq_status tq_quantize_kv_append(const tq_kv_cache* cache, const uint16_t* k_new,
                                const uint16_t* v_new, int32_t n_new,
                                const int32_t* write_pos, int32_t* status,
                                void* stream);

/* tq_quantize_kv_append with rotation: flags TQ_ROTATE_K / TQ_ROTATE_V rotate
 * each new K / V row by H (see the rotation flags above) before it is
 * quantized; the rotation is fused into the same kernel (no extra pass over
 * the rows).  Rotated rows are fp16_rne(fp32 transform), then quantized by the
 * rule above.  Other flag bits: TQ_ERR_UNSUPPORTED. */
tq_status tq_quantize_kv_append_ex(const tq_kv_cache* cache, const uint16_t* k_new,
                                   const uint16_t* v_new, int32_t n_new,
                                   const int32_t* write_pos, uint32_t flags,
                                   int32_t* status, void* stream);

/* out[r] = fp16_rne(H x[r]) for `rows` rows of `dim` fp16 values (dim 64, 128
 * or 256; device pointers, 16-byte aligned; out may equal x).  H as for the
 * rotation flags.  rows = 0 launches nothing. */
tq_status tq_hadamard_rotate(const uint16_t* x, int64_t rows, int32_t dim,
                             uint16_t* out, void* stream);

/* ------------------------------------------------------------ paged cache --
 * Bytes of a page pool for these sizes (the six arrays, each 256-aligned),
 * 0 for invalid sizes.  Host-only. */
size_t tq_paged_kv_cache_bytes(int32_t num_pages, int32_t num_kv_heads, int32_t head_dim,
                               int32_t group_size, int32_t bits, int32_t page_tokens);

/* Fill *cache with the arrays carved from `base` (device, 256-byte aligned,
 * tq_paged_kv_cache_bytes long) and the given block table.  Host-only. */
tq_status tq_paged_kv_cache_carve(tq_paged_kv_cache* cache, void* base, const int32_t* block_table,
                                  int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t group_size, int32_t bits, int32_t page_tokens,
                                  int32_t num_pages, int32_t max_pages_per_seq);

/* tq_quantize_kv_append_ex into a paged cache (rows through the block table). */
tq_status tq_paged_quantize_kv_append(const tq_paged_kv_cache* cache, const uint16_t* k_new,
                                      const uint16_t* v_new, int32_t n_new,
                                      const int32_t* write_pos, uint32_t flags,
                                      int32_t* status, void* stream);

/* tq_sdpa_int4_decode_ex / tq_decode_step_ex over a paged cache: the same
 * arithmetic and, for chunk >= 128, the same split plan as the contiguous
 * cache (runs start on page-aligned tile boundaries; smaller chunks are
 * raised to the tile), so the results are identical to a contiguous cache
 * holding the same rows.  Tensor-core path only. */
tq_status tq_paged_sdpa_int4_decode(const tq_paged_kv_cache* cache, const uint16_t* q,
                                    int32_t num_q_heads, const int32_t* seq_lens,
                                    int32_t max_seq_len, float attn_scale, int32_t chunk,
                                    uint32_t flags, void* workspace, size_t workspace_bytes,
                                    uint16_t* out, int32_t* status, void* stream);
tq_status tq_paged_decode_step(const tq_paged_kv_cache* cache, const uint16_t* k_new,
                               const uint16_t* v_new, int32_t n_new, const int32_t* write_pos,
                               const uint16_t* q, int32_t num_q_heads, const int32_t* seq_lens,
                               int32_t max_seq_len, float attn_scale, int32_t chunk, uint32_t flags,
                               void* workspace, size_t workspace_bytes, uint16_t* out,
                               int32_t* status, void* stream);

/* ------------------------------------------------------------ host buffers --
 * tq_decode_step_ex with the step's inputs and output in host memory: copies
 * q [batch][num_q_heads][head_dim] and k_new / v_new [batch][Hkv][n_new][D]
 * (fp16, host; page-locked for the copies to be asynchronous) into `staging`
 * (device, 256-byte aligned, tq_host_staging_bytes long), runs the step, and
 * copies the fp16 output back to h_out (host).  Everything is queued on
 * `stream` in one call (no host synchronisation): h_out holds the result once
 * the stream has reached it.  write_pos, seq_lens, workspace and status stay
 * device-side, as for tq_decode_step_ex.  The call a serving loop makes once
 * per step when its activations live on the host.  When all four host buffers
 * are page-locked and mapped (cudaHostAlloc, torch pin_memory) the kernels
 * read and write them in place (GPU-addressable host memory, NVLink-C2C on
 * Grace-Blackwell) and `staging` is not touched. */
size_t tq_host_staging_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t n_new);
tq_status tq_decode_step_host(const tq_kv_cache* cache, const uint16_t* h_k_new,
                              const uint16_t* h_v_new, int32_t n_new, const int32_t* write_pos,
                              const uint16_t* h_q, int32_t num_q_heads, const int32_t* seq_lens,
                              int32_t max_seq_len, float attn_scale, int32_t chunk, uint32_t flags,
                              void* workspace, size_t workspace_bytes, void* staging,
                              size_t staging_bytes, uint16_t* h_out, int32_t* status, void* stream);

/* Workspace bytes tq_sdpa_int4_decode needs for these sizes (an upper bound
 * that does not depend on the device).  Host-only. */
size_t tq_sdpa_workspace_bytes(int32_t batch, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t max_seq_len, int32_t chunk);

/* Fused int4 decode attention (Sq = 1, GQA).
 * q:        fp16 [batch][num_q_heads][head_dim]; query head h reads KV head
 *           h / (num_q_heads / num_kv_heads)  (num_q_heads / num_kv_heads <= 8)
 * seq_lens: device int32 [batch]; sequence b attends to cache rows
 *           [0, seq_lens[b]); 0 gives an all-zero output row
 * max_seq_len: host bound on seq_lens (1 <= max_seq_len <= capacity); sizes the grid
 * attn_scale: multiplies q.k (1/sqrt(head_dim) for Llama, 1.0 for Gemma)
 * chunk:    split-K chunk in tokens (multiple of 16; TQ_DEFAULT_CHUNK = 512).
 *           The sequence is split into balanced runs, one per CTA, of whole
 *           units of min(chunk, pipeline tile) tokens (the tile is 384 tokens
 *           for contiguous int4 caches at head_dim 128, else 128 tokens when a
 *           token's codes take under 128 bytes, 64 otherwise); each run
 *           keeps one running softmax
 *           state and the runs' states are merged by a log-sum-exp reduce
 *           (tq_sdpa_int4_reduce; with at most 8 runs in a grid of one wave the
 *           runs of each (sequence, kv head) form one thread-block cluster and
 *           merge in phase 1 with the reduce's operations, bit for bit the same
 *           output).  The result is the same as merging one state per chunk
 *           (see tq_sdpa_int4_partial with chunks_per_split = 1).
 * workspace: device scratch (256-byte aligned) of at least
 *           tq_sdpa_workspace_bytes(...) bytes holding the fp32 partial states,
 *           room for a rotated query and, for batches whose grid spans several
 *           waves, the device-computed dispatch order of the runs (longest
 *           first); contents on entry are ignored.
 * out:      fp16 [batch][num_q_heads][head_dim], round-to-nearest-even.
 * Accumulation is fp32; result within 2e-3 abs / 1e-3 rel-L2 of fp64 attention
 * over the dequantised cache. */
tq_status tq_sdpa_int4_decode(const tq_kv_cache* cache, const uint16_t* q,
                              int32_t num_q_heads, const int32_t* seq_lens,
                              int32_t max_seq_len, float attn_scale,
                              int32_t chunk, void* workspace,
                              size_t workspace_bytes, uint16_t* out,
                              int32_t* status, void* stream);

/* Same as tq_sdpa_int4_decode with an explicit implementation choice. */
tq_status tq_sdpa_int4_decode_impl(const tq_kv_cache* cache, const uint16_t* q,
                                   int32_t num_q_heads, const int32_t* seq_lens,
                                   int32_t max_seq_len, float attn_scale,
                                   int32_t chunk, void* workspace,
                                   size_t workspace_bytes, uint16_t* out,
                                   int32_t* status, tq_impl impl, void* stream);

/* One decode step: quantize-on-store of the new tokens, then fused int4 decode
 * attention over the cache that now holds them ("turboquant-llama3.170B"
 * README, decode-step listing: quantize K,V to int4, then fused sdpa_int4).
 * Arguments as tq_quantize_kv_append and tq_sdpa_int4_decode (tensor-core
 * path); results identical to calling the two in order on `stream`.  The
 * decode launch may start while the append still runs and waits for it only
 * in the CTAs whose runs read an appended row.  seq_lens must already count
 * the new tokens (typically write_pos[b] + n_new). */
tq_status tq_decode_step(const tq_kv_cache* cache, const uint16_t* k_new,
                         const uint16_t* v_new, int32_t n_new,
                         const int32_t* write_pos, const uint16_t* q,
                         int32_t num_q_heads, const int32_t* seq_lens,
                         int32_t max_seq_len, float attn_scale, int32_t chunk,
                         void* workspace, size_t workspace_bytes,
                         uint16_t* out, int32_t* status, void* stream);

/* Decode over a cache written with rotation flags (the same flags as its
 * appends): TQ_ROTATE_K rotates the query (into the workspace) before phase
 * 1; TQ_ROTATE_V applies H to the merged output before its fp16 rounding.
 * Otherwise as tq_sdpa_int4_decode / tq_decode_step (a rotated step appends
 * its rows inside the decode kernel like an unrotated one, rotating each row
 * across the lanes that hold it). */
tq_status tq_sdpa_int4_decode_ex(const tq_kv_cache* cache, const uint16_t* q,
                                 int32_t num_q_heads, const int32_t* seq_lens,
                                 int32_t max_seq_len, float attn_scale, int32_t chunk,
                                 uint32_t flags, void* workspace, size_t workspace_bytes,
                                 uint16_t* out, int32_t* status, void* stream);
tq_status tq_decode_step_ex(const tq_kv_cache* cache, const uint16_t* k_new,
                            const uint16_t* v_new, int32_t n_new,
                            const int32_t* write_pos, const uint16_t* q,
                            int32_t num_q_heads, const int32_t* seq_lens,
                            int32_t max_seq_len, float attn_scale, int32_t chunk,
                            uint32_t flags, void* workspace, size_t workspace_bytes,
                            uint16_t* out, int32_t* status, void* stream);

/* The split plan tq_sdpa_int4_decode uses on the current device: *n_splits
 * runs per (sequence, kv head), the longest *max_run_tokens tokens long.
 * Host-side query (reads device attributes). */
tq_status tq_sdpa_plan(const tq_kv_cache* cache, int32_t num_q_heads,
                       int32_t max_seq_len, int32_t chunk, tq_impl impl,
                       int32_t* n_splits, int32_t* max_run_tokens);

/* The split plan rule itself, without a device: the runs per (sequence, kv
 * head) for `batch` sequences of up to `max_seq_len` tokens, `num_kv_heads`
 * kv heads, runs made of whole units of min(chunk, tile_tokens) tokens, on a
 * device that holds `resident_ctas` phase-1 CTAs at once (tq_sdpa_plan passes
 * the SM count x the CTAs per SM and the kernel's tile: 384 tokens for a
 * contiguous int4 cache at head_dim 128, one CTA per SM; else 128 tokens when a
 * token's codes take under 128 bytes, 64 otherwise).  Picks the run count
 * n <= min(units, 2048 / (batch * num_kv_heads)) that minimises, with
 * W = ceil(batch * num_kv_heads * n / resident_ctas) waves,
 *   W * (ceil(units / n) * unit + 2 * tile_tokens) + R,
 * R = tile_tokens for the reduce, or 0 when `merge` is nonzero and the
 * decode merges the runs itself (n = 1, or n <= 8 with W = 1: one
 * thread-block cluster per sequence and kv head); the fewest runs on a tie.
 * tq_sdpa_plan passes merge = 1 (0 for the CUDA-core implementation); steps
 * with TQ_ROTATE_V or TQ_STEP_ADVANCE, whose reduce has other work, plan with
 * merge = 0.  Chunk and tile_tokens must be positive multiples of 16 and every
 * count positive (TQ_ERR_SHAPE), the outputs non-null (TQ_ERR_NULL).  Pure
 * host arithmetic. */
tq_status tq_split_plan(int32_t batch, int32_t num_kv_heads, int32_t max_seq_len,
                        int32_t chunk, int32_t tile_tokens, int32_t resident_ctas,
                        int32_t merge, int32_t* n_splits, int32_t* max_run_tokens);

/* Split-K phase 1 alone ("turboquant-llama3.170B" README, split-K paragraph:
 * Phase 1 = partial attention over 512-token chunks processed in parallel).
 * Each part covers `chunks_per_split` consecutive chunks (1 = one state per
 * chunk, the pages' form), np = ceil(ceil(max_seq_len / chunk) /
 * chunks_per_split); or, with chunks_per_split = 0, the runs
 * tq_sdpa_int4_decode uses (np = n_splits of tq_sdpa_plan).  fp32 outputs:
 *   part_m   [batch][num_q_heads][np]  max over the part of the scaled score
 *            (natural-log units; -inf for an empty part)
 *   part_l   [batch][num_q_heads][np]  sum of exp(score - m)  (0 if empty)
 *   part_acc [batch][num_q_heads][np][head_dim]  sum of exp(score - m) * v
 * Parts past seq_lens[b] are empty.  Arrays must hold np entries per (b, h). */
tq_status tq_sdpa_int4_partial(const tq_kv_cache* cache, const uint16_t* q,
                               int32_t num_q_heads, const int32_t* seq_lens,
                               int32_t max_seq_len, float attn_scale,
                               int32_t chunk, int32_t chunks_per_split,
                               float* part_m, float* part_l, float* part_acc,
                               int32_t* status, tq_impl impl, void* stream);

/* Expand rows [0, n_rows) of every (sequence, KV head) of the cache into fp16
 * K and V, k_out / v_out [batch][num_kv_heads][n_rows][head_dim] (device,
 * caller-owned, 16-byte aligned):
 *   value = fp16_rne(fp32(scale * code + bias))
 * (one fp32 rounding -- the product is exact -- then RNE to binary16).  This
 * is the float cache of the dequantize-then-attend decode that the fused
 * kernel replaces ("Fused int4 Attention for Gemma 4 31B on Apple Silicon",
 * What I Built Instead); it is here as that comparison point, not as a step of
 * the fused path.  Errors: TQ_ERR_NULL, TQ_ERR_SHAPE (n_rows < 0),
 * TQ_ERR_CAPACITY (n_rows > capacity), TQ_ERR_ALIGN, plus the cache checks.
 * n_rows = 0 launches nothing. */
tq_status tq_dequantize_kv(const tq_kv_cache* cache, int32_t n_rows,
                           uint16_t* k_out, uint16_t* v_out, void* stream);

/* Split-K phase 2 alone ("Phase 2 (reduce)" of the same paragraph): per (b, h),
 *   M = max over parts with l > 0 of m,  w_c = exp(m_c - M),
 *   out = sum_c w_c acc_c / sum_c w_c l_c   (fp16, RNE; all-empty rows -> 0).
 * Inputs laid out as tq_sdpa_int4_partial writes them, n_parts per (b, h),
 * 1 <= n_parts <= 8192. */
tq_status tq_sdpa_int4_reduce(const float* part_m, const float* part_l,
                              const float* part_acc, int32_t batch,
                              int32_t num_q_heads, int32_t head_dim,
                              int32_t n_parts, uint16_t* out, void* stream);

/* Size of the library-owned device array tq_sdpa_int4_decode_noalloc keeps its
 * partial states in (per GPU that loads the library, held until exit). */
#define TQ_NOALLOC_SCRATCH_BYTES (4u << 20)

/* Fused int4 decode attention for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point.  It is
 * tq_sdpa_int4_decode (tensor-core path) without the workspace argument: the
 * split-K partial states go to a fixed TQ_NOALLOC_SCRATCH_BYTES device array
 * inside the library, so the call allocates nothing.  Meant for callers that
 * have no allocator at hand or may not use one: code in host callbacks or
 * other paths where cudaMalloc is forbidden, plugins of frameworks that own
 * all device memory, plain C programs that link only this library.
 *   - Same arguments, layouts and results as tq_sdpa_int4_decode, bit for
 *     bit (the same plan and kernels).  One difference in speed: batches
 *     whose grid spans several waves run in grid order, without the
 *     longest-run-first dispatch pass of the workspace decode.
 *   - Requests whose partial states do not fit the array return
 *     TQ_ERR_WORKSPACE before any launch.  They need, with P = batch *
 *     num_q_heads * n_splits (n_splits as tq_sdpa_plan reports) and A(n) = n
 *     rounded up to a multiple of 256,  2 * A(4 P) + 4 P * head_dim  bytes
 *     (m and l, each 256-byte aligned, then acc).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is kept per device and looked
 *     up again when the device has a new context (after cudaDeviceReset);
 *     make that next call before any capture too.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents; nothing in it needs clearing (each call writes every element
 *     it reads), but calls that overlap on the GPU (other streams, other host
 *     threads) race on it and may return wrong results: serialise them. */
tq_status tq_sdpa_int4_decode_noalloc(const tq_kv_cache* cache, const uint16_t* q,
                                      int32_t num_q_heads, const int32_t* seq_lens,
                                      int32_t max_seq_len, float attn_scale,
                                      int32_t chunk, uint16_t* out,
                                      int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */

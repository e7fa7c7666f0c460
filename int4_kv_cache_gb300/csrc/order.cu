// order.cu -- dispatch order of the split-K runs of a batched decode whose
// grid spans several waves: longest run first.
//
// The runs of sequence b are [run_begin(s), run_begin(s + 1)) clipped to its
// length, which only the device knows.  Launched in grid order, the runs of
// the batch's last sequences start in the last wave whatever their length,
// and a long one started late decides the decode time; dispatched longest
// first (the longest-processing-time rule), the short and empty runs fill
// the tail instead.  One CTA counts the runs per length in tiles, takes the
// descending prefix sum of the counts and scatters the run indices, each with
// its sequence's length (the decode CTA then needs no second read); the order
// within one length is not fixed, which does not change any result (every
// run writes its own partial state).
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kOrderThreads = 1024;
constexpr int kOrderKeys = 1024;  // run lengths in tiles, the last key holding all longer runs

__device__ __forceinline__ int run_key(const OrderParams& p, int item) {
    const int b = item / p.n_splits, s = item % p.n_splits;
    const int len = min(max(__ldg(p.seq_lens + b), 0), p.max_seq_len);
    const int lo = run_begin(s, p.units, p.n_splits, p.unit_tokens);
    const int hi = min(run_begin(s + 1, p.units, p.n_splits, p.unit_tokens), len);
    const int tiles = hi > lo ? (hi - lo + p.tile_tokens - 1) / p.tile_tokens : 0;
    return min(tiles, kOrderKeys - 1);
}

__global__ void __launch_bounds__(kOrderThreads) order_runs_kernel(const OrderParams p) {
    __shared__ int count[kOrderKeys];
    __shared__ int warp_sum[kOrderThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = p.batch * p.n_splits;
    pdl_wait_primary();  // the lengths may come from the kernel before
    for (int k = tid; k < kOrderKeys; k += kOrderThreads) count[k] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kOrderThreads) atomicAdd(&count[run_key(p, i)], 1);
    __syncthreads();
    // start[k] = number of runs longer than k: an inclusive scan over the keys
    // in descending order (thread t holds key K - 1 - t), minus its own count
    const int key = kOrderKeys - 1 - tid;
    const int c = count[key];
    int v = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    if (lane == 31) warp_sum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += u;
        }
        warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sum[warp - 1] : 0) + v - c;
    count[key] = before;  // each key is owned by one thread
    __syncthreads();
    pdl_launch_dependents();
    for (int i = tid; i < n; i += kOrderThreads) {
        const int b = i / p.n_splits, raw = __ldg(p.seq_lens + b);
        if ((raw < 0 || raw > p.max_seq_len) && i % p.n_splits == 0 && p.status != nullptr)
            atomicOr(p.status, TQ_DEV_SEQ_LEN);
        p.order[atomicAdd(&count[run_key(p, i)], 1)] = make_int2(i, min(max(raw, 0), p.max_seq_len));
    }
}

static_assert(kOrderKeys == kOrderThreads, "one key per thread in the scan");

}  // namespace

cudaError_t launch_order_runs(const OrderParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kOrderThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, order_runs_kernel, p);
}

}  // namespace tq

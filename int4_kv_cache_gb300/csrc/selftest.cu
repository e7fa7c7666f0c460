// selftest.cu -- a diagnostic of the bounded pipeline wait the decode kernels
// use (mbar_wait_bounded): one CTA completes a bulk copy into shared memory
// and waits for it, then waits on an mbarrier that nothing arrives at, with a
// short limit.  The wait gives up, the CTA records TQ_DEV_TIMEOUT in the
// status word and returns; no copy is in flight when it leaves, so the
// context stays usable.  The same status path ends a decode CTA whose stage
// never fills.
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kSelftestBytes = 1024;

__global__ void wait_timeout_kernel(const uint4* __restrict__ src, int32_t* status, uint64_t limit_ns,
                                    uint32_t* copied) {
    __shared__ __align__(128) uint4 buf[kSelftestBytes / 16];
    __shared__ uint64_t bar_copy, bar_never;
    if (threadIdx.x == 0) {
        mbar_init(&bar_copy, 1);
        mbar_init(&bar_never, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar_copy, kSelftestBytes);
        bulk_load(buf, src, kSelftestBytes, &bar_copy, policy_evict_first());
    }
    // the copy completes: every thread sees it land
    const bool landed = mbar_wait_bounded(&bar_copy, 0, limit_ns);
    // phase 0 of bar_never never completes (its one arrival never comes)
    const bool arrived = mbar_wait_bounded(&bar_never, 0, limit_ns);
    if (threadIdx.x == 0) {
        if (!arrived && status != nullptr) atomicOr(status, TQ_DEV_TIMEOUT);
        uint32_t sum = 0;
        if (landed)
            for (int i = 0; i < kSelftestBytes / 16; ++i) sum += buf[i].x + buf[i].y + buf[i].z + buf[i].w;
        *copied = landed ? sum : 0xFFFFFFFFu;
    }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(const void* src, int32_t* status, uint64_t limit_ns, uint32_t* copied,
                                         cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(static_cast<const uint4*>(src), status, limit_ns, copied);
    return cudaGetLastError();
}

}  // namespace tq

// rotate.cu -- the Hadamard rotation of fp16 rows (query vectors, or keys
// before a separate quantize): out = fp16_rne((1/sqrt(n)) H_n x) with the fp32
// fast transform of tq_hadamard.cuh.  One warp per row; every row access is a
// contiguous, coalesced 4/8/16-byte load or store per lane.
#include "tq_device.cuh"
#include "tq_hadamard.cuh"
#include "tq_internal.h"

namespace tq {

namespace {

constexpr int kRotThreads = 256;

template <int E>
__global__ void __launch_bounds__(kRotThreads) rotate_rows_kernel(const uint16_t* x, long long rows, uint16_t* out,
                                                                  float scale) {
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * (kRotThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;  // the whole warp
    struct alignas(2 * E) Vec {
        uint16_t h[E];
    };
    const Vec in = reinterpret_cast<const Vec*>(x + row * (32 * E))[lane];
    float v[E];
    halves_to_floats<E>(in.h, v);
    hadamard_warp<E>(v, lane, scale);
    Vec o;
    floats_to_halves<E>(v, o.h);
    reinterpret_cast<Vec*>(out + row * (32 * E))[lane] = o;
}

}  // namespace

cudaError_t launch_rotate_rows(const uint16_t* x, long long rows, int dim, uint16_t* out, float scale,
                               cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const long long blocks = (rows + kRotThreads / 32 - 1) / (kRotThreads / 32);
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks));
    switch (dim) {
        case 64: rotate_rows_kernel<2><<<grid, kRotThreads, 0, stream>>>(x, rows, out, scale); break;
        case 128: rotate_rows_kernel<4><<<grid, kRotThreads, 0, stream>>>(x, rows, out, scale); break;
        case 256: rotate_rows_kernel<8><<<grid, kRotThreads, 0, stream>>>(x, rows, out, scale); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace tq

// Measured dense INT8 tensor peak of this part (diagnostics, not the GEMM).
//
// sm_103a has no integer tcgen05 MMA, so the GPU's INT8 tensor rate is that of
// the warp-level mma.sync s8 instruction.  This kernel issues nothing else:
// each warp runs `iters` rounds of eight independent m16n8k32 s8 x s8 -> s32
// MMAs on register operands (no memory traffic), and writes one checksum so
// that the work is kept.  The caller times the launch; the operation count is
// blocks x 8 warps x iters x 8 x (2 x 16 x 8 x 32).
#include <cuda_runtime.h>
#include <stdint.h>

#include "q4k_internal.h"

namespace q4k {
namespace {

constexpr int kPeakThreads = 256;
constexpr int kChains = 8;

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__global__ void __launch_bounds__(kPeakThreads) peak_s8_kernel(int64_t iters, int* sink) {
    const uint32_t seed = threadIdx.x * 2654435761u + blockIdx.x;
    uint32_t a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = seed * (i + 3) ^ 0x01010101u;
#pragma unroll
    for (int i = 0; i < 2; ++i) b[i] = seed * (i + 7) ^ 0x02020202u;
    int acc[kChains][4] = {};
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) mma_s8(acc[c], a, b);
    }
    int s = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += acc[c][0] ^ acc[c][1] ^ acc[c][2] ^ acc[c][3];
    if (s == 0x7FFFFFFF) sink[blockIdx.x] = s;   // practically never: keeps the work without a store per thread
    if (threadIdx.x == 0) sink[blockIdx.x] = s;
}

}  // namespace

cudaError_t launch_peak_s8(int64_t blocks, int64_t iters, int* sink, cudaStream_t s) {
    peak_s8_kernel<<<static_cast<unsigned>(blocks), kPeakThreads, 0, s>>>(iters, sink);
    return cudaGetLastError();
}

}  // namespace q4k

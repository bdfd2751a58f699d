// Activation quantization into 32-element q8 blocks.
//
// "34 · r31 — q-major sda scale-read repack", §1: each q8 block of the
// activations carries an f16 scale d and an i16 ssum (the sum of its q8
// values); the pair feeds the two-term rescale.  Rounding (the page prints
// none): d = RN32(amax/127), inv = RN32(127/amax),
// qa = clamp(rint_half_even(RN32(x*inv)), -127, 127), d_a = RN16(d);
// blocks with amax < 2^-120 are zero blocks.
//
// The public q8 form (q8_rows_kernel): one thread per block, its eight 16-B
// loads in flight together, amax and ssum without shuffles; a warp takes 32
// consecutive blocks of one token (4 KB of contiguous fp32).  Its small
// batches and the q8-to-operand conversion use an 8-lane group per block, the
// GEMM operand form (act_quant_kernel) a lane pair per block.  HBM-bound: 4 B
// read per element, 1 B (public q8) or 2 B (GEMM operand) written per element
// plus a few bytes per block.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4k_internal.h"
#include "q4k_layout.h"
#include "q4k_ptx.cuh"
#include "q8_operand.cuh"
#include "q8_rule.cuh"

namespace q4k {
namespace {

constexpr int kThreadsPerBlock = 256;

// An 8-lane group per 32-element block (each lane one float4, amax and ssum
// by shuffles within the group): eight times the threads of the one-thread
// form, for batches too small to fill the GPU with one thread per block.
constexpr unsigned kFull = 0xFFFFFFFFu;

struct LaneQ8 {
    int q[4];
    int ssum;       // whole block
    __half da;      // whole block
};

__device__ __forceinline__ LaneQ8 quantize_lane(float4 v) {
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1, 8));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2, 8));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4, 8));
    const Q8Scale sc = q8_scale(amax);
    LaneQ8 r;
    const float xs[4] = {v.x, v.y, v.z, v.w};
    int s = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        r.q[i] = q8_code(xs[i], sc);
        s += r.q[i];
    }
    s += __shfl_xor_sync(kFull, s, 1, 8);
    s += __shfl_xor_sync(kFull, s, 2, 8);
    s += __shfl_xor_sync(kFull, s, 4, 8);
    r.ssum = s;
    r.da = sc.da;
    return r;
}

// The q8 block of 32 consecutive fp32 values at src (16-byte aligned): codes,
// d_a and ssum, by the rule in the header of this file (fp32, this order;
// amax and ssum do not depend on the order of their terms).
struct BlockQ8 {
    int q[32];
    int ssum;
    __half da;
};

__device__ __forceinline__ BlockQ8 quantize_block(const float* __restrict__ src) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(src) + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
    }
    float amax = fabsf(v[0]);
#pragma unroll
    for (int i = 1; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const Q8Scale sc = q8_scale(amax);
    BlockQ8 b;
    b.ssum = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        b.q[i] = q8_code(v[i], sc);
        b.ssum += b.q[i];
    }
    b.da = sc.da;
    return b;
}

// Public SoA output, 8-lane groups (small batches).
__global__ void __launch_bounds__(kThreadsPerBlock) q8_rows_lanes_kernel(const float* __restrict__ x, int64_t m,
                                                                         int64_t k, int64_t ldx,
                                                                         int8_t* __restrict__ q8,
                                                                         uint16_t* __restrict__ da,
                                                                         int16_t* __restrict__ ssum) {
    griddep_launch_dependents();   // programmatic dependent launch (see q8_rows_kernel)
    griddep_wait();
    const int64_t kc = k / 32;
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t grp = gid >> 3;
    const int j = static_cast<int>(gid & 7);
    // whole 8-lane groups stay in range together: m*kc*8 is a multiple of 8
    const bool in = grp < m * kc;
    const int64_t t = in ? grp / kc : 0, c = in ? grp % kc : 0;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (in) v = __ldg(reinterpret_cast<const float4*>(x + t * ldx + c * 32 + 4 * j));
    const LaneQ8 r = quantize_lane(v);
    if (!in) return;
    const uint32_t packed = (static_cast<uint32_t>(r.q[0]) & 0xFFu) | ((static_cast<uint32_t>(r.q[1]) & 0xFFu) << 8) |
                            ((static_cast<uint32_t>(r.q[2]) & 0xFFu) << 16) |
                            ((static_cast<uint32_t>(r.q[3]) & 0xFFu) << 24);
    *reinterpret_cast<uint32_t*>(q8 + t * k + c * 32 + 4 * j) = packed;
    if (j == 0) {
        da[t * kc + c] = __half_as_ushort(r.da);
        ssum[t * kc + c] = static_cast<int16_t>(r.ssum);
    }
}

// Public SoA output: q8 [m][k], da f16 [m][kc], ssum i16 [m][kc].
__global__ void __launch_bounds__(kThreadsPerBlock) q8_rows_kernel(const float* __restrict__ x, int64_t m, int64_t k,
                                                                   int64_t ldx, int8_t* __restrict__ q8,
                                                                   uint16_t* __restrict__ da,
                                                                   int16_t* __restrict__ ssum) {
    // launched with programmatic dependent launch: let the next kernel (the
    // small-M product) start staging its weights, and wait for the previous
    // one (which may still read q8/da/ssum, or have written x) to finish
    griddep_launch_dependents();
    griddep_wait();
    const int64_t kc = k / 32, kg = (kc + 31) / 32;   // 32-block groups per token
    const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t t = wid / kg, c = (wid % kg) * 32 + (threadIdx.x & 31);
    if (t >= m || c >= kc) return;
    const BlockQ8 b = quantize_block(x + t * ldx + c * 32);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = (static_cast<uint32_t>(b.q[4 * i]) & 0xFFu) | ((static_cast<uint32_t>(b.q[4 * i + 1]) & 0xFFu) << 8) |
               ((static_cast<uint32_t>(b.q[4 * i + 2]) & 0xFFu) << 16) |
               ((static_cast<uint32_t>(b.q[4 * i + 3]) & 0xFFu) << 24);
    uint4* dst = reinterpret_cast<uint4*>(q8 + t * k + c * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    da[t * kc + c] = __half_as_ushort(b.da);
    ssum[t * kc + c] = static_cast<int16_t>(b.ssum);
}

__device__ __forceinline__ void write_operand(int64_t t, int64_t c, int j, int64_t m, int64_t k, int64_t kc,
                                              const int (&q)[4], __half da, int ssum, uint16_t* __restrict__ xq,
                                              float* __restrict__ dat, __nv_bfloat16* __restrict__ e) {
    uint2 w;
    w.x = code_pair(q[0], q[1]);
    w.y = code_pair(q[2], q[3]);
    *reinterpret_cast<uint2*>(xq + t * k + c * 32 + 4 * j) = w;
    if (j == 0) {
        dat[((t >> 7) * kc + c) * 128 + (t & 127)] = __half2float(da);
        __nv_bfloat16 hi, lo;
        split_e(da, ssum, hi, lo);
        e[t * kc + c] = hi;
        e[(m + t) * kc + c] = lo;
    }
}

// GEMM operand form (see q4k_layout.h; fp16 codes) from fp32 activations.  A
// lane pair takes one 32-k block (quantize_pair_block in q8_operand.cuh, the
// routine the GEMM's in-kernel quantization runs too: 16 values a lane, its
// four 16-B loads in flight together; amax and ssum need one shuffle), and a warp 16 consecutive
// blocks of one token (2 KB of fp32; k is a multiple of 256, so the last warp
// of a token may hold 8).  Against an 8-lane group per block this halves the
// shuffles and doubles the bytes each lane has in flight: 12% less time at
// 2048 tokens.  The input is read once, so it is loaded with the evict-first
// hint and leaves L2 to the operand the GEMM reads next.
__global__ void __launch_bounds__(kThreadsPerBlock) act_quant_kernel(const float* __restrict__ x, int64_t m,
                                                                     int64_t mp, int64_t k, int64_t ldx,
                                                                     uint16_t* __restrict__ xq,
                                                                     float* __restrict__ dat,
                                                                     __nv_bfloat16* __restrict__ e) {
    griddep_launch_dependents();   // programmatic dependent launch (see q8_rows_kernel)
    griddep_wait();
    const int64_t kc = k / 32, wpt = (kc + 15) / 16;   // warps per token
    const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t = wid / wpt, c = (wid % wpt) * 16 + (lane >> 1);
    if (t >= mp) return;   // whole warps: t is the same across the warp
    quantize_pair_block(x, ldx, m, k, kc, t, c, lane & 1, c < kc, xq, dat, e);
}

// GEMM operand form from the public q8 SoA ([m][ldq] int8, da, ssum [m][kc]).
__global__ void __launch_bounds__(kThreadsPerBlock) act_from_q8_kernel(const int8_t* __restrict__ q8,
                                                                       const uint16_t* __restrict__ da,
                                                                       const int16_t* __restrict__ ssum, int64_t m,
                                                                       int64_t mp, int64_t k, int64_t ldq,
                                                                       uint16_t* __restrict__ xq,
                                                                       float* __restrict__ dat,
                                                                       __nv_bfloat16* __restrict__ e) {
    griddep_launch_dependents();   // programmatic dependent launch (see q8_rows_kernel)
    griddep_wait();
    const int64_t kc = k / 32;
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t grp = gid >> 3;
    const int j = static_cast<int>(gid & 7);
    if (grp >= mp * kc) return;
    const int64_t t = grp / kc, c = grp % kc;
    if (t >= m) {
        if (j == 0) dat[((t >> 7) * kc + c) * 128 + (t & 127)] = 0.0f;
        return;
    }
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(q8 + t * ldq + c * 32 + 4 * j));
    int q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = static_cast<int>(static_cast<int8_t>((w >> (8 * i)) & 0xFFu));
    const __half dh = __ushort_as_half(da[t * kc + c]);
    write_operand(t, c, j, m, k, kc, q, dh, static_cast<int>(ssum[t * kc + c]), xq, dat, e);
}

inline unsigned grid_for(int64_t threads) {
    return static_cast<unsigned>((threads + kThreadsPerBlock - 1) / kThreadsPerBlock);
}

}  // namespace

cudaError_t launch_q8_quantize_rows(const float* x, int64_t m, int64_t k, int64_t ldx, int8_t* q8, uint16_t* da,
                                    int16_t* ssum, cudaStream_t s) {
    const int64_t blocks = m * (k / 32);
    if (blocks == 0) return cudaSuccess;
    // fewer blocks than about 64 CTAs of one thread each: 8 lanes per block
    if (blocks < 64 * kThreadsPerBlock)
        return launch_pdl(q8_rows_lanes_kernel, dim3(grid_for(blocks * 8)), dim3(kThreadsPerBlock), 0, s, x, m, k, ldx,
                          q8, da, ssum);
    const int64_t threads = m * ((k / 32 + 31) / 32) * 32;   // a warp per 32 blocks of a token
    return launch_pdl(q8_rows_kernel, dim3(grid_for(threads)), dim3(kThreadsPerBlock), 0, s, x, m, k, ldx, q8, da,
                      ssum);
}

cudaError_t launch_act_quantize(const float* x, int64_t m, int64_t k, int64_t ldx, void* ws, cudaStream_t s) {
    const ActLayout L(m, k);
    const int64_t mp = align_up(m, kTileM);
    const int64_t threads = mp * ((k / 32 + 15) / 16) * 32;   // a warp per 16 blocks of a token
    if (threads == 0) return cudaSuccess;
    uint8_t* b = static_cast<uint8_t*>(ws);
    uint16_t* xq = reinterpret_cast<uint16_t*>(b + L.xq);
    float* dat = reinterpret_cast<float*>(b + L.da);
    __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(b + L.e);
    return launch_pdl(act_quant_kernel, dim3(grid_for(threads)), dim3(kThreadsPerBlock), 0, s, x, m, mp, k, ldx, xq,
                      dat, e);
}

cudaError_t launch_act_from_q8(const int8_t* q8, const uint16_t* da, const int16_t* ssum, int64_t m, int64_t k,
                               int64_t ldq, void* ws, cudaStream_t s) {
    const ActLayout L(m, k);
    const int64_t mp = align_up(m, kTileM);
    const int64_t threads = mp * (k / 32) * 8;
    if (threads == 0) return cudaSuccess;
    uint8_t* b = static_cast<uint8_t*>(ws);
    uint16_t* xq = reinterpret_cast<uint16_t*>(b + L.xq);
    float* dat = reinterpret_cast<float*>(b + L.da);
    __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(b + L.e);
    return launch_pdl(act_from_q8_kernel, dim3(grid_for(threads)), dim3(kThreadsPerBlock), 0, s, q8, da, ssum, m, mp,
                      k, ldq, xq, dat, e);
}

}  // namespace q4k

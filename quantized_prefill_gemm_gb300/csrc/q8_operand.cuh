// The GEMM's activation operand (q4k_layout.h, ActLayout) for one 32-k block
// of one token, computed by a lane pair: the one routine behind both the
// separate quantization pass (act_quant.cu) and the GEMM's own in-kernel
// quantization (gemm.cu), so that the two write the same bits.
//
// The q8 rule itself (q8_rule.cuh) is "34 · r31 — q-major sda scale-read
// repack", §1: per block an f16 d_a and the sum of the codes.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "q8_rule.cuh"

namespace q4k {

// Two q8 codes as an exact fp16 pair (the GEMM operand of both weight formats).
__device__ __forceinline__ uint32_t code_pair(int q0, int q1) {
    const __half2 pr = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
    return *reinterpret_cast<const uint32_t*>(&pr);
}

// E = d_a * ssum (exact in fp32: an 11-bit by <= 12-bit product) split into
// two bf16 terms hi + lo with |E - hi - lo| <= 2^-16 |E|.
__device__ __forceinline__ void split_e(__half da, int ssum, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    const float e = __fmul_rn(__half2float(da), static_cast<float>(ssum));
    hi = __float2bfloat16_rn(e);
    lo = __float2bfloat16_rn(__fsub_rn(e, __bfloat162float(hi)));
}

// Block c of token t, by a lane pair: the lane with half = lane & 1 takes the
// 16 values 16*half .. 16*half + 15.  pair_load issues its four 16-byte loads
// (several pairs' loads can be in flight before the first pair_finish);
// pair_finish combines amax and ssum over the pair with one shuffle each and
// writes the operand.  All 32 lanes of the warp must call pair_finish
// together (the shuffles); `in` false marks a lane pair with no block.  For a
// padding token (m <= t < mp) the pair writes d_a = 0 only.  x is read once,
// with the evict-first hint.
__device__ __forceinline__ void pair_load(const float* __restrict__ x, int64_t ldx, int64_t m, int64_t t, int64_t c,
                                          int half, bool in, float (&v)[16]) {
    const bool live = in && t < m;
    const float4* src = reinterpret_cast<const float4*>(x + (live ? t * ldx + c * 32 + 16 * half : 0));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 f = live ? __ldcs(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
    }
}

__device__ __forceinline__ void pair_finish(const float (&v)[16], int64_t m, int64_t k, int64_t kc, int64_t t,
                                            int64_t c, int half, bool in, uint16_t* __restrict__ xq,
                                            float* __restrict__ dat, __nv_bfloat16* __restrict__ e) {
    constexpr unsigned kAll = 0xFFFFFFFFu;
    float amax = fabsf(v[0]);
#pragma unroll
    for (int i = 1; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 1));
    const Q8Scale sc = q8_scale(amax);
    uint32_t w[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q0 = q8_code(v[2 * i], sc), q1 = q8_code(v[2 * i + 1], sc);
        sum += q0 + q1;
        w[i] = code_pair(q0, q1);
    }
    sum += __shfl_xor_sync(kAll, sum, 1);
    if (!in) return;
    float* dslot = dat + ((t >> 7) * kc + c) * 128 + (t & 127);
    if (t >= m) {   // padding token of the last 128-token tile: scale 0
        if (half == 0) *dslot = 0.0f;
        return;
    }
    uint4* dst = reinterpret_cast<uint4*>(xq + t * k + c * 32 + 16 * half);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    if (half == 0) {
        *dslot = __half2float(sc.da);
        __nv_bfloat16 hi, lo;
        split_e(sc.da, sum, hi, lo);
        e[t * kc + c] = hi;
        e[(m + t) * kc + c] = lo;
    }
}

__device__ __forceinline__ void quantize_pair_block(const float* __restrict__ x, int64_t ldx, int64_t m, int64_t k,
                                                    int64_t kc, int64_t t, int64_t c, int half, bool in,
                                                    uint16_t* __restrict__ xq, float* __restrict__ dat,
                                                    __nv_bfloat16* __restrict__ e) {
    float v[16];
    pair_load(x, ldx, m, t, c, half, in, v);
    pair_finish(v, m, k, kc, t, c, half, in, xq, dat, e);
}

}  // namespace q4k

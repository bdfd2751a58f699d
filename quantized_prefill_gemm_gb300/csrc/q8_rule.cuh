// The q8 block rule, in one place for every kernel that quantizes activations
// (the bit-exactness of q8 codes, d_a and ssum across kernels rests on them
// all taking these same fp32 operations in this order).
//
// "34 · r31 — q-major sda scale-read repack", §1: each block of 32
// consecutive activations of one token carries an f16 scale d_a and the sum of
// its q8 codes.  The pages give no rounding rule; the one used here, from the
// block's absolute maximum amax (fp32):
//   live = amax >= 2^-120     (below it 127 / amax overflows: a zero block)
//   d    = RN(amax / 127),    inv = RN(127 / amax)
//   qa   = live ? clamp(rint_even(RN(x * inv)), -127, 127) : 0
//   d_a  = RN16(live ? d : 0)
// amax and ssum = sum(qa) do not depend on the order of their terms.
#pragma once
#include <cuda_fp16.h>

namespace q4k {

struct Q8Scale {
    float inv;    // RN(127 / amax)
    __half da;    // RN16(d), +0 for a zero block
    bool live;
};

__device__ __forceinline__ Q8Scale q8_scale(float amax) {
    Q8Scale s;
    s.live = amax >= 0x1p-120f;
    const float d = __fdiv_rn(amax, 127.0f);
    s.inv = __fdiv_rn(127.0f, amax);
    s.da = __float2half_rn(s.live ? d : 0.0f);
    return s;
}

__device__ __forceinline__ int q8_code(float x, const Q8Scale& s) {
    const int q = max(-127, min(127, __float2int_rn(__fmul_rn(x, s.inv))));
    return s.live ? q : 0;
}

}  // namespace q4k

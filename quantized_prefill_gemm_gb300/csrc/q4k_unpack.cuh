// Quant unpacking shared by the small-M kernels and the GEMM's converters.
#pragma once
#include <stdint.h>

namespace q4k {

// 4-bit quants of one 8-k group (one packed word) -> two words of 4 bytes in
// k order.  In the packed word the nibble at bits 4j is k = 2j and the nibble
// at bits 16 + 4j is k = 2j + 1.
__device__ __forceinline__ void unpack_group(uint32_t w, uint32_t& k0123, uint32_t& k4567) {
    const uint32_t a = w & 0x000F000Fu;           // bytes 0, 2: k0, k1
    const uint32_t b = (w >> 4) & 0x000F000Fu;    // bytes 0, 2: k2, k3
    const uint32_t c = (w >> 8) & 0x000F000Fu;    // k4, k5
    const uint32_t e = (w >> 12) & 0x000F000Fu;   // k6, k7
    k0123 = __byte_perm(a, b, 0x6420);
    k4567 = __byte_perm(c, e, 0x6420);
}

// Q6_K: signed bytes q - 32 of one 8-k group from its low-nibble word and the
// high-bit word shifted to the group (2-bit fields at the group's nibble
// positions).  u = q ^ 32 is q - 32 in 6-bit two's complement: low nibble and
// high bits are put back together and bit 5 is copied into bits 6 and 7.
__device__ __forceinline__ void unpack_q6(uint32_t lo, uint32_t hi, uint32_t& v0123, uint32_t& v4567) {
    uint32_t l0, l1, h0, h1;
    unpack_group(lo, l0, l1);
    unpack_group(hi & 0x33333333u, h0, h1);
    const uint32_t u0 = l0 | (h0 << 4), u1 = l1 | (h1 << 4);   // 6-bit u per byte
    v0123 = u0 | ((u0 & 0x20202020u) * 6u);
    v4567 = u1 | ((u1 & 0x20202020u) * 6u);
}

}  // namespace q4k

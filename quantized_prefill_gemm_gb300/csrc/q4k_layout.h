// Internal buffer layouts of the library (host and device code share them).
//
// Packed weights (q4k_pack_weights -> q4k_gemm), for n od rows and k inputs,
// nt = n/128 row tiles, kc = k/32 chunks, ksb = k/256 super-blocks:
//   nib  [nt][kc][128][16 B]  4-bit quants of one (od row, chunk): 4 words, word i
//                              holds k = 8i..8i+7 of the chunk; inside a word the
//                              nibble at bits 4j (j < 4) is k = 8i+2j and the
//                              nibble at bits 16+4j is k = 8i+2j+1, so masking
//                              with 0x000F000F after a shift by 4j gives the
//                              k-consecutive pair (8i+2j, 8i+2j+1).
//   sc   [nt][kc][128]  u8    6-bit sub-block scale sc
//   dsb  [nt][ksb][128] f32   super-block scale d
//   ndm  [2][n][kc]     bf16  -(dmin*m) split into hi = bf16(v) (plane 0) and
//                              lo = bf16(v - hi) (plane 1)
//   mq   [nt][kc][128]  u8    6-bit sub-block min m        (small-M path)
//   dmn  [nt][ksb][128] f32   super-block dmin             (small-M path)
//
// Activation workspace (q4k_act_quantize / q4k_act_from_q8 -> q4k_gemm), for m
// tokens, mp = m rounded up to 128:
//   xq   [m][k]            f16   qa as an exact fp16 integer in [-127, 127]
//   da   [mp/128][kc][128] f32   d_a (exact f16 value), zero for padding tokens
//   e    [2][m][kc]        bf16  E = d_a*ssum (exact in fp32) split into
//                                 hi = bf16(E) (plane 0), lo = bf16(E - hi) (plane 1)
//   part [kMaxSplitUnits][8][32][64] f32  partial tiles of the GEMM's k-split
//                                 tail: unit (tail tile, part), slice (2 x row
//                                 quadrant + column half), row, column
//   flag [mp/128]          u64   in-kernel quantization (q4k_gemm from fp32):
//                                 per 128-token tile, the call's tag in bits
//                                 16-63 and the count of its quantized slices
//                                 in bits 0-15 (gemm.cu)
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace q4k {

constexpr int64_t kAlign = 1024;
constexpr int64_t kTileM = 128;   // tokens per GEMM tile (TMEM lanes)
constexpr int64_t kTileN = 128;   // output features per GEMM tile
constexpr int64_t kMaxSplitUnits = 160;   // k-split work units of one GEMM launch (>= its grid)

inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

struct PackedLayout {
    int64_t nib, sc, dsb, ndm, mq, dmn, total;
    PackedLayout(int64_t n, int64_t k) {
        const int64_t kc = k / 32, ksb = k / 256;
        nib = 0;
        sc = align_up(nib + n * k / 2, kAlign);
        dsb = align_up(sc + n * kc, kAlign);
        ndm = align_up(dsb + n * ksb * 4, kAlign);
        mq = align_up(ndm + 2 * n * kc * 2, kAlign);
        dmn = align_up(mq + n * kc, kAlign);
        total = align_up(dmn + n * ksb * 4, kAlign);
    }
};

// Q6_K weights for the small-M path (q6k_pack_weights -> q6k_gemm), for n
// rows and k inputs, nt = n/128, kc = k/32, ksb = k/256.  With u = q ^ 32 (the
// 6-bit two's complement of q - 32):
//   lo  [nt][kc][128][16 B]  low 4 bits of u, nibbles arranged as in nib above
//   hi  [nt][kc][128][8 B]   bits 4-5 of u: word 0 holds 8-k groups 0 and 1,
//                             word 1 groups 2 and 3; the group's 2-bit fields
//                             sit at the group's nibble positions (first group
//                             of the word in bits 0-1, second in bits 2-3)
//   sc  [nt][kc][128][2]  i8  the scales of the chunk's two 16-weight sub-blocks
//   dsb [nt][ksb][128]    f32 super-block scale d
struct Q6Layout {
    int64_t lo, hi, sc, dsb, total;
    Q6Layout(int64_t n, int64_t k) {
        const int64_t kc = k / 32, ksb = k / 256;
        lo = 0;
        hi = align_up(lo + n * k / 2, kAlign);
        sc = align_up(hi + n * k / 4, kAlign);
        dsb = align_up(sc + n * kc * 2, kAlign);
        total = align_up(dsb + n * ksb * 4, kAlign);
    }
};

struct ActLayout {
    int64_t xq, da, e, part, flag, total;
    ActLayout(int64_t m, int64_t k) {
        const int64_t kc = k / 32, mp = align_up(m, kTileM);
        xq = 0;
        da = align_up(xq + m * k * 2, kAlign);
        e = align_up(da + mp * kc * 4, kAlign);
        part = align_up(e + 2 * m * kc * 2, kAlign);
        flag = align_up(part + kMaxSplitUnits * 8 * 32 * 64 * 4, kAlign);
        total = align_up(flag + (mp / kTileM) * 8, kAlign);
    }
};

}  // namespace q4k

// Small-M (decode-sized) product with the packed weights streamed through a
// shared-memory ring: m <= 4 tokens with Q4_K or Q6_K weights (dp4a), and
// 5..16 tokens of q8 input with Q4_K weights (integer mma.sync).
//
// The arithmetic is the small-M kernels' (per 32-k chunk an exact integer dot
// product of the 4- or 6-bit quants with the q8 codes, then the block
// rescale of "34 · r31 — q-major sda scale-read repack", §1-§2); what differs
// is how the weights reach the SMs and how few instructions a weight costs.
// At one token the product is one pass over the weights: it is bound by the
// bytes in flight from HBM, by the SM's instruction rate per weight byte, and
// by the part of each launch that streams nothing (launch, first loads, the
// row sums, the tail).  So:
//
//   - two CTAs of 256 threads per SM (grid G = min(row groups, 2 x SMs)); CTA
//     b owns the 16-row groups b, b + G, b + 2G, ..., every group over all of
//     k, so no partial sum leaves the CTA, and the CTAs working at the same
//     time read neighbouring slices of the same 128-row records;
//   - the CTA's weights flow through a ring of R stages (a few super-blocks
//     of one group each) filled with 16-byte cp.async copies whose source
//     addresses are fixed per thread up to a per-stage offset, R-1 stages in
//     flight while one is consumed; their completion is the hardware's
//     wait_group, so no thread spins on a flag;
//   - launched with programmatic dependent launch: as soon as a CTA is
//     resident it asks L2 for its 1/G share of the launch's weights (a
//     prefetch hint: it cannot change what a later load returns) and only
//     then waits for the kernel before it, so the weights come from HBM while
//     that kernel finishes.  Every read of the ring or of the activations
//     comes after the wait.
//
// Q4_K without unpacking: in a packed quant word the nibbles of k = 0,4,1,5
// sit at bits 0, 8, 16, 24 and those of k = 2,6,3,7 at bits 4, 12, 20, 28
// (the word layout of the packed format), so w & 0x0F0F0F0F is a byte vector
// dp4a takes as it is, and w & 0xF0F0F0F0 one of 16 x the other nibbles
// (unsigned bytes), against the activations staged with each 8-byte group
// reordered to k = 0,4,1,5,2,6,3,7.  The integer dot product is the same sum
// in another order.
//
// Thread t takes row r = t % 16 of the group and the stage's chunks
// (t / 16) * I .. + I - 1 (I = 4 for Q4_K, 2 for Q6_K; one super-block); a
// row's sums are added over its 16 threads (a shuffle, then 8 warps' partials
// in shared memory in a fixed order) at the end of each group and stored.
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <algorithm>

#include "q4k_internal.h"
#include "q4k_gemv.h"
#include "q4k_ptx.cuh"
#include "q8_rule.cuh"
#include "q4k_unpack.cuh"

namespace q4k {
namespace {

constexpr int kRows = 16;      // od rows per group
constexpr int kThreads = 256;  // 16 chunk columns x 16 rows
constexpr size_t kStreamMaxSmem = 220 * 1024;
constexpr uint32_t kLowNibbles = 0x0F0F0F0Fu;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Ask L2 for this CTA's share of one packed array: its 4 KB pages b, b + G,
// b + 2G, ... (over the grid, the whole array), issued by the first warp.
__device__ __forceinline__ void prefetch_pages(const void* base, int64_t bytes, int b, int G) {
    const int64_t pages = (bytes + 4095) >> 12;
    for (int64_t pg = b + static_cast<int64_t>(G) * (threadIdx.x & 31); pg < pages; pg += 32 * static_cast<int64_t>(G)) {
        const int64_t off = pg << 12;
        prefetch_l2(static_cast<const uint8_t*>(base) + off, static_cast<uint32_t>(bytes - off < 4096 ? bytes - off : 4096));
    }
}

// ------------------------------------------------------------ formats --
// dp4a of unsigned bytes a with signed bytes b
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// One warp-level integer MMA, D = A (16 x 32 unsigned bytes) * B (32 x 8
// signed bytes) + 0, with the fragment layout of mma.m16n8k32: lane l holds
// A rows l/4 and l/4 + 8 at k-slots 4(l%4)..+3 (a0, a1) and 16 + 4(l%4)..+3
// (a2, a3), B column l/4 at the same two slot groups (b0, b1), and D rows l/4
// (d0, d1) and l/4 + 8 (d2, d3) at columns 2(l%4), 2(l%4) + 1.
__device__ __forceinline__ void mma_u8s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%10,%11,%12,%13};"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0), "r"(0), "r"(0), "r"(0));
}

// The same with k = 16 (m16n8k16): lane l holds A rows l/4 and l/4 + 8 at
// k-slots 4(l%4)..+3 (a0, a1) and B column l/4 at the same slots (b0).
__device__ __forceinline__ void mma_u8s8_k16(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%8,%9,%10};"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(a0), "r"(a1), "r"(b0), "r"(0), "r"(0), "r"(0), "r"(0));
}

// Q6_K quants q = u ^ 32 (0..63, unsigned bytes) of one packed 8-k group from
// its low-nibble word and its 2-bit high fields hf (at the group's nibble
// positions, low two bits of each nibble), in the two permuted byte orders
// of the Q4_K masks: q0 for k = 0,4,1,5, q1 for k = 2,6,3,7.  hf ^ 0x22..
// flips bit 5 of u in both.
__device__ __forceinline__ void q6_bytes(uint32_t lo, uint32_t hf, uint32_t& q0, uint32_t& q1) {
    const uint32_t hx = hf ^ 0x22222222u;
    q0 = (lo & kLowNibbles) | ((hx << 4) & 0x30303030u);
    q1 = ((lo >> 4) & kLowNibbles) | (hx & 0x30303030u);
}

// Q4_K: nib 16 B, sc 1 B, m 1 B per (row, chunk); d, dmin fp32 per (row, sb).
// A stage is kSb super-blocks (8 in use); a thread takes kSb / 2 chunks of
// one super-block.
template <int kSb>
struct Q4StreamT {
    static constexpr int kStageSb = kSb;
    static constexpr int kItems = kSb / 2;   // 8 kSb chunks over 16 chunk columns
    static constexpr bool kPermuted = true;   // activations staged in the nibble order
    static constexpr bool kHalfSums = false;  // staged: d_a * ssum
    static constexpr bool kMma = true;        // 8 and 16 tokens on the tensor cores (compute_mma)
    static constexpr int kMmaChunks = 8;      // chunks a warp takes per stage in that form: one super-block
    static constexpr uint32_t kNib = 0;
    static constexpr uint32_t kSc = kNib + 8 * kStageSb * kRows * 16;
    static constexpr uint32_t kMq = kSc + 8 * kStageSb * kRows;
    static constexpr uint32_t kD = kMq + 8 * kStageSb * kRows;
    static constexpr uint32_t kDmin = kD + kStageSb * kRows * 4;
    static constexpr uint32_t kSlot = kDmin + kStageSb * kRows * 4;
    // What thread t copies of every stage (152 kSb 16-byte pieces): the
    // quants of chunks t/16 + 16h (h < kSb/2), row slice t%16, and for
    // t < 24 kSb one piece of the sc, m, d or dmin records.  Only the stage
    // bases move.
    static constexpr int kScPieces = 8 * kSb;   // sc (and m) pieces of a stage: one per chunk
    static constexpr int kDPieces = 4 * kSb;    // d (and dmin) pieces: four per super-block
    struct Copier {
        const uint8_t* q;   // this thread's first quant piece of the next stage
        const uint8_t* x;   // its scale piece, or null
        uint32_t qdst, xdst;
        int qu, xu;         // chunk of the first quant piece; chunk (sc, m) or super-block (d, dmin) of the scale piece
        bool xsb;           // the scale piece is per super-block
        uint32_t xstep;

        __device__ void init() {
            const int t = threadIdx.x;
            qu = t >> 4;
            qdst = kNib + 16 * t;
            x = nullptr;
            xu = 0;
            xsb = false;
            xstep = 0;
            xdst = 0;
            if (t < 2 * kScPieces) {
                xu = t % kScPieces;
                xdst = (t < kScPieces ? kSc : kMq) + 16 * xu;
                xstep = 8 * kStageSb * 128;
            } else if (t < 2 * kScPieces + 2 * kDPieces) {
                const int q = (t - 2 * kScPieces) % kDPieces;
                xu = q >> 2;
                xsb = true;
                xdst = (t < 2 * kScPieces + kDPieces ? kD : kDmin) + 16 * q;
                xstep = kStageSb * 128 * 4;
            }
        }
        // first stage of the group of rows r0 .. r0 + 15 of tile nt
        __device__ void group(const GemvParams& p, int64_t nt, int r0) {
            const int t = threadIdx.x;
            q = p.nib + ((nt * p.kc + qu) * 128 + r0 + (t & 15)) * 16;
            if (t < 2 * kScPieces) {
                x = (t < kScPieces ? p.sc : p.mq) + (nt * p.kc + xu) * 128 + r0;
            } else if (t < 2 * kScPieces + 2 * kDPieces) {
                const float* b = t < 2 * kScPieces + kDPieces ? p.dsb : p.dmn;
                x = reinterpret_cast<const uint8_t*>(b + (nt * p.ksb + xu) * 128 + r0) + 16 * (t & 3);
            }
        }
        // the stage of ns super-blocks into the ring slot at shared address slot; then on to the next stage
        __device__ void issue(uint32_t slot, int ns) {
#pragma unroll
            for (int h = 0; h < kSb / 2; ++h)
                if (qu + 16 * h < 8 * ns) cp_async16(slot + qdst + 4096 * h, q + 32768 * h);
            if (x && xu < (xsb ? ns : 8 * ns)) cp_async16(slot + xdst, x);
            q += 8 * kStageSb * 2048;
            if (x) x += xstep;
        }
    };
    __device__ static void prefetch(const GemvParams& p, int b, int G) {
        const int64_t n = p.n;
        prefetch_pages(p.nib, n * p.k / 2, b, G);
        prefetch_pages(p.sc, n * p.kc, b, G);
        prefetch_pages(p.mq, n * p.kc, b, G);
        prefetch_pages(p.dsb, n * p.ksb * 4, b, G);
        prefetch_pages(p.dmn, n * p.ksb * 4, b, G);
    }
    // Row r, chunks j0 .. j0 + kItems - 1 of the stage (global chunks c0 ..):
    //   acc += d * sum_c d_a * (sc * J) - dmin * sum_c m * (d_a * ssum)
    // J = J_lo + J_hi / 16: the low nibbles as they sit, the high nibbles
    // masked in place (16 x their value, unsigned bytes); both sums exact.
    template <int M>
    __device__ static void compute(const uint8_t* sl, int j0, int r, int c0, const int8_t* act, const float2* xs,
                                   int m, int k, int kc, float (&acc)[M]) {
        float P[M], Z[M];
#pragma unroll
        for (int t = 0; t < M; ++t) {
            P[t] = 0.0f;
            Z[t] = 0.0f;
        }
#pragma unroll
        for (int e = 0; e < kItems; ++e) {
            const int j = j0 + e, c = c0 + e;
            const uint4 qw = *reinterpret_cast<const uint4*>(sl + kNib + (j * kRows + r) * 16);
            const int sc = sl[kSc + j * kRows + r];
            const float mv = static_cast<float>(sl[kMq + j * kRows + r]);
            const int l0 = static_cast<int>(qw.x & kLowNibbles), l1 = static_cast<int>(qw.y & kLowNibbles);
            const int l2 = static_cast<int>(qw.z & kLowNibbles), l3 = static_cast<int>(qw.w & kLowNibbles);
            const uint32_t h0 = qw.x & ~kLowNibbles, h1 = qw.y & ~kLowNibbles;
            const uint32_t h2 = qw.z & ~kLowNibbles, h3 = qw.w & ~kLowNibbles;
#pragma unroll
            for (int t = 0; t < M; ++t) {
                if (t < m) {
                    const int4* a = reinterpret_cast<const int4*>(act + (static_cast<int64_t>(c) * M + t) * 32);
                    const int4 a0 = a[0], a1 = a[1];
                    int Jl = __dp4a(l0, a0.x, 0);
                    int Jh = dp4a_us(h0, a0.y, 0);
                    Jl = __dp4a(l1, a0.z, Jl);
                    Jh = dp4a_us(h1, a0.w, Jh);
                    Jl = __dp4a(l2, a1.x, Jl);
                    Jh = dp4a_us(h2, a1.y, Jh);
                    Jl = __dp4a(l3, a1.z, Jl);
                    Jh = dp4a_us(h3, a1.w, Jh);
                    const int J = Jl + (Jh >> 4);
                    const float2 s = xs[c * M + t];   // d_a, d_a * ssum (both exact in fp32)
                    P[t] = fmaf(s.x, static_cast<float>(sc * J), P[t]);   // sc * J < 2^22: exact
                    Z[t] = fmaf(s.y, mv, Z[t]);
                }
            }
        }
        const float d = reinterpret_cast<const float*>(sl + kD)[(j0 >> 3) * kRows + r];
        const float dmin = reinterpret_cast<const float*>(sl + kDmin)[(j0 >> 3) * kRows + r];
#pragma unroll
        for (int t = 0; t < M; ++t) acc[t] = fmaf(-dmin, Z[t], fmaf(d, P[t], acc[t]));
    }
    // 8 or 16 tokens on the tensor cores (mma.sync m16n8k32, u8 x s8): warp w
    // takes super-block w of the stage for all 16 rows of the group.  The A
    // operand is 16 x the quants: for word i of a row, k-slots 4i..4i+3 hold
    // its low nibbles shifted up and 16 + 4i..+3 its high nibbles masked in
    // place; the B operand is the activations staged in the same permuted
    // order (an 8-byte load gives both slot groups).  So D = 16 J exactly.
    // acc[4 mi + e]: rows l/4 (e < 2) and l/4 + 8, tokens 8 mi + 2(l%4) + e%2.
    template <int M>
    __device__ static void compute_mma(const uint8_t* sl, int w, int lane, int c0, const int8_t* act, const float2* xs,
                                       int k, int kc, float (&acc)[M / 2]) {
        constexpr int kN = M / 8;   // n8 blocks of tokens
        const int g = lane >> 2, q = lane & 3;
        float P[4 * kN], Z[4 * kN];
#pragma unroll
        for (int i = 0; i < 4 * kN; ++i) {
            P[i] = 0.0f;
            Z[i] = 0.0f;
        }
#pragma unroll 2
        for (int jj = 0; jj < 8; ++jj) {
            const int j = 8 * w + jj, c = c0 + jj;
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(sl + kNib + (j * kRows + g) * 16 + 4 * q);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(sl + kNib + (j * kRows + g + 8) * 16 + 4 * q);
            const uint32_t a0 = (w0 << 4) & ~kLowNibbles, a1 = (w1 << 4) & ~kLowNibbles;
            const uint32_t a2 = w0 & ~kLowNibbles, a3 = w1 & ~kLowNibbles;
            const int sc0 = sl[kSc + j * kRows + g], sc1 = sl[kSc + j * kRows + g + 8];
            const float m0 = static_cast<float>(sl[kMq + j * kRows + g]);
            const float m1 = static_cast<float>(sl[kMq + j * kRows + g + 8]);
#pragma unroll
            for (int mi = 0; mi < kN; ++mi) {
                const uint2 b = *reinterpret_cast<const uint2*>(act + (static_cast<int64_t>(c) * M + 8 * mi + g) * 32 + 8 * q);
                int d[4];
                mma_u8s8(d, a0, a1, a2, a3, b.x, b.y);
                const float4 s01 = *reinterpret_cast<const float4*>(xs + c * M + 8 * mi + 2 * q);   // tokens 2q, 2q + 1
                const float2 s0 = make_float2(s01.x, s01.y), s1 = make_float2(s01.z, s01.w);
                // d / 16 = J exactly; sc * J < 2^22
                P[4 * mi + 0] = fmaf(s0.x, static_cast<float>(sc0 * (d[0] >> 4)), P[4 * mi + 0]);
                P[4 * mi + 1] = fmaf(s1.x, static_cast<float>(sc0 * (d[1] >> 4)), P[4 * mi + 1]);
                P[4 * mi + 2] = fmaf(s0.x, static_cast<float>(sc1 * (d[2] >> 4)), P[4 * mi + 2]);
                P[4 * mi + 3] = fmaf(s1.x, static_cast<float>(sc1 * (d[3] >> 4)), P[4 * mi + 3]);
                Z[4 * mi + 0] = fmaf(s0.y, m0, Z[4 * mi + 0]);
                Z[4 * mi + 1] = fmaf(s1.y, m0, Z[4 * mi + 1]);
                Z[4 * mi + 2] = fmaf(s0.y, m1, Z[4 * mi + 2]);
                Z[4 * mi + 3] = fmaf(s1.y, m1, Z[4 * mi + 3]);
            }
        }
        const float* dv = reinterpret_cast<const float*>(sl + kD) + w * kRows;
        const float* nv = reinterpret_cast<const float*>(sl + kDmin) + w * kRows;
        const float d0 = dv[g], d1 = dv[g + 8], n0 = nv[g], n1 = nv[g + 8];
#pragma unroll
        for (int mi = 0; mi < kN; ++mi) {
            acc[4 * mi + 0] = fmaf(-n0, Z[4 * mi + 0], fmaf(d0, P[4 * mi + 0], acc[4 * mi + 0]));
            acc[4 * mi + 1] = fmaf(-n0, Z[4 * mi + 1], fmaf(d0, P[4 * mi + 1], acc[4 * mi + 1]));
            acc[4 * mi + 2] = fmaf(-n1, Z[4 * mi + 2], fmaf(d1, P[4 * mi + 2], acc[4 * mi + 2]));
            acc[4 * mi + 3] = fmaf(-n1, Z[4 * mi + 3], fmaf(d1, P[4 * mi + 3], acc[4 * mi + 3]));
        }
    }
};

using Q4Stream = Q4StreamT<8>;

// Q6_K: lo 16 B, hi 8 B, the two i8 scales 2 B per (row, chunk); d fp32 per
// (row, sb).  A stage is 4 super-blocks; a thread takes 2 chunks of one.
struct Q6Stream {
    static constexpr int kStageSb = 4;
    static constexpr int kItems = 2;
    static constexpr bool kPermuted = true;
    static constexpr bool kHalfSums = true;   // staged: the two half-chunk code sums
    static constexpr bool kMma = true;        // 8 and 16 tokens on the tensor cores (compute_mma)
    static constexpr int kMmaChunks = 4;      // chunks a warp takes per stage in that form: half a super-block
    static constexpr uint32_t kLo = 0;
    static constexpr uint32_t kHi = kLo + 8 * kStageSb * kRows * 16;
    static constexpr uint32_t kSc = kHi + 8 * kStageSb * kRows * 8;
    static constexpr uint32_t kD = kSc + 8 * kStageSb * kRows * 2;
    static constexpr uint32_t kSlot = kD + kStageSb * kRows * 4;

    // What thread t copies of every stage (848 16-byte pieces): the low
    // nibbles of chunks t/16 and t/16 + 16, row slice t%16; the high bits of
    // chunk t/8, slice t%8; and for t < 80 one piece of the scale pairs or d.
    struct Copier {
        const uint8_t* lo;
        const uint8_t* hi;
        const uint8_t* x;   // scale-pair or d piece, or null
        uint32_t xdst;
        int lu, hu, xu;     // chunks of the lo and hi pieces; chunk or super-block of the x piece
        bool xsb;
        uint32_t xstep;

        __device__ void init() {
            const int t = threadIdx.x;
            lu = t >> 4;
            hu = t >> 3;
            x = nullptr;
            xu = 0;
            xsb = false;
            xstep = 0;
            xdst = 0;
            if (t < 64) {
                xu = t >> 1;
                xdst = kSc + 16 * t;
                xstep = 8 * kStageSb * 128 * 2;
            } else if (t < 80) {
                const int q = t - 64;
                xu = q >> 2;
                xsb = true;
                xdst = kD + 16 * q;
                xstep = kStageSb * 128 * 4;
            }
        }
        __device__ void group(const GemvParams& p, int64_t nt, int r0) {
            const int t = threadIdx.x;
            lo = p.nib + ((nt * p.kc + lu) * 128 + r0 + (t & 15)) * 16;
            hi = p.q6hi + ((nt * p.kc + hu) * 128 + r0) * 8 + 16 * (t & 7);
            if (t < 64)
                x = p.sc + ((nt * p.kc + xu) * 128 + r0) * 2 + 16 * (t & 1);
            else if (t < 80)
                x = reinterpret_cast<const uint8_t*>(p.dsb + (nt * p.ksb + xu) * 128 + r0) + 16 * (t & 3);
        }
        __device__ void issue(uint32_t slot, int ns) {
            const int t = threadIdx.x;
            if (lu < 8 * ns) cp_async16(slot + kLo + 16 * t, lo);
            if (lu + 16 < 8 * ns) cp_async16(slot + kLo + 16 * t + 4096, lo + 32768);
            if (hu < 8 * ns) cp_async16(slot + kHi + 16 * t, hi);
            if (x && xu < (xsb ? ns : 8 * ns)) cp_async16(slot + xdst, x);
            lo += 8 * kStageSb * 2048;
            hi += 8 * kStageSb * 1024;
            if (x) x += xstep;
        }
    };
    __device__ static void prefetch(const GemvParams& p, int b, int G) {
        const int64_t n = p.n;
        prefetch_pages(p.nib, n * p.k / 2, b, G);
        prefetch_pages(p.q6hi, n * p.k / 4, b, G);
        prefetch_pages(p.sc, n * p.kc * 2, b, G);
        prefetch_pages(p.dsb, n * p.ksb * 4, b, G);
    }
    // I = sc_0 * sum_{k<16} (q-32) qa + sc_1 * sum_{k>=16} (q-32) qa (|I| < 2^24, exact in fp32), as
    // sc_h * (sum q qa - 32 X_h) with q the unsigned 6-bit quants and X_h the half's code sum
    template <int M>
    __device__ static void compute(const uint8_t* sl, int j0, int r, int c0, const int8_t* act, const float2* xs,
                                   int m, int k, int kc, float (&acc)[M]) {
        float P[M];
#pragma unroll
        for (int t = 0; t < M; ++t) P[t] = 0.0f;
#pragma unroll
        for (int e = 0; e < kItems; ++e) {
            const int j = j0 + e, c = c0 + e;
            const uint4 lo = *reinterpret_cast<const uint4*>(sl + kLo + (j * kRows + r) * 16);
            const uint2 hi = *reinterpret_cast<const uint2*>(sl + kHi + (j * kRows + r) * 8);
            const uint32_t scp = *reinterpret_cast<const uint16_t*>(sl + kSc + (j * kRows + r) * 2);
            uint32_t q[8];
            q6_bytes(lo.x, hi.x, q[0], q[1]);
            q6_bytes(lo.y, hi.x >> 2, q[2], q[3]);
            q6_bytes(lo.z, hi.y, q[4], q[5]);
            q6_bytes(lo.w, hi.y >> 2, q[6], q[7]);
            const int sc0 = static_cast<int>(static_cast<int8_t>(scp & 0xFFu));
            const int sc1 = static_cast<int>(static_cast<int8_t>(scp >> 8));
#pragma unroll
            for (int t = 0; t < M; ++t) {
                if (t < m) {
                    const int4* a = reinterpret_cast<const int4*>(act + (static_cast<int64_t>(c) * M + t) * 32);
                    const int4 a0 = a[0], a1 = a[1];
                    int J0 = dp4a_us(q[0], a0.x, 0);
                    int J1 = dp4a_us(q[4], a1.x, 0);
                    J0 = dp4a_us(q[1], a0.y, J0);
                    J1 = dp4a_us(q[5], a1.y, J1);
                    J0 = dp4a_us(q[2], a0.z, J0);
                    J1 = dp4a_us(q[6], a1.z, J1);
                    J0 = dp4a_us(q[3], a0.w, J0);
                    J1 = dp4a_us(q[7], a1.w, J1);
                    const float2 s = xs[c * M + t];
                    const int xp = __float_as_int(s.y);
                    const int X0 = (xp << 16) >> 16, X1 = xp >> 16;
                    const int I = sc0 * (J0 - 32 * X0) + sc1 * (J1 - 32 * X1);
                    P[t] = fmaf(s.x, static_cast<float>(I), P[t]);
                }
            }
        }
        const float d = reinterpret_cast<const float*>(sl + kD)[(j0 >> 3) * kRows + r];
#pragma unroll
        for (int t = 0; t < M; ++t) acc[t] = fmaf(d, P[t], acc[t]);
    }
    // 8 or 16 tokens on the tensor cores: warp w takes chunks 4w..4w+3 of the
    // stage (half of super-block w/2) for all 16 rows, two m16n8k16 MMAs per
    // chunk, one per 16-weight half (its own scale).  The A operand is the
    // unsigned q = u ^ 32: for half h, k-slots 4i..4i+3 hold word 2h + i/2 of
    // the row in the low-nibble (i even) or high-nibble (i odd) byte order of
    // the Q4_K masks; B is the activations staged in the same order.  Then
    // I = sc_h * (D_h - 32 X_h) summed over the halves, exact.
    // acc[4 mi + e]: rows l/4 (e < 2) and l/4 + 8, tokens 8 mi + 2(l%4) + e%2.
    template <int M>
    __device__ static void compute_mma(const uint8_t* sl, int w, int lane, int c0, const int8_t* act, const float2* xs,
                                       int k, int kc, float (&acc)[M / 2]) {
        constexpr int kN = M / 8;
        const int g = lane >> 2, q = lane & 3;
        const int wq = q >> 1;            // this lane's word within a half
        const bool odd = (q & 1) != 0;    // high-nibble byte order
        float P[4 * kN];
#pragma unroll
        for (int i = 0; i < 4 * kN; ++i) P[i] = 0.0f;
#pragma unroll 2
        for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * w + jj, c = c0 + jj;
            uint32_t a[2][2];   // [half][row g, row g + 8]
            int sc[2][2];       // [row][half]
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int row = g + 8 * rr;
                const uint32_t* lw = reinterpret_cast<const uint32_t*>(sl + kLo + (j * kRows + row) * 16);
                const uint2 hw = *reinterpret_cast<const uint2*>(sl + kHi + (j * kRows + row) * 8);
                const uint32_t scp = *reinterpret_cast<const uint16_t*>(sl + kSc + (j * kRows + row) * 2);
                sc[rr][0] = static_cast<int>(static_cast<int8_t>(scp & 0xFFu));
                sc[rr][1] = static_cast<int>(static_cast<int8_t>(scp >> 8));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t q0, q1;
                    q6_bytes(lw[2 * h + wq], (h ? hw.y : hw.x) >> (2 * wq), q0, q1);
                    a[h][rr] = odd ? q1 : q0;
                }
            }
#pragma unroll
            for (int mi = 0; mi < kN; ++mi) {
                const int8_t* bt = act + (static_cast<int64_t>(c) * M + 8 * mi + g) * 32 + 4 * q;
                int d0[4], d1[4];
                mma_u8s8_k16(d0, a[0][0], a[0][1], *reinterpret_cast<const uint32_t*>(bt));
                mma_u8s8_k16(d1, a[1][0], a[1][1], *reinterpret_cast<const uint32_t*>(bt + 16));
                const float4 s01 = *reinterpret_cast<const float4*>(xs + c * M + 8 * mi + 2 * q);   // tokens 2q, 2q + 1
                const int xp0 = __float_as_int(s01.y), xp1 = __float_as_int(s01.w);
                const int x00 = (xp0 << 16) >> 16, x01 = xp0 >> 16, x10 = (xp1 << 16) >> 16, x11 = xp1 >> 16;
                P[4 * mi + 0] = fmaf(s01.x, static_cast<float>(sc[0][0] * (d0[0] - 32 * x00) + sc[0][1] * (d1[0] - 32 * x01)),
                                     P[4 * mi + 0]);
                P[4 * mi + 1] = fmaf(s01.z, static_cast<float>(sc[0][0] * (d0[1] - 32 * x10) + sc[0][1] * (d1[1] - 32 * x11)),
                                     P[4 * mi + 1]);
                P[4 * mi + 2] = fmaf(s01.x, static_cast<float>(sc[1][0] * (d0[2] - 32 * x00) + sc[1][1] * (d1[2] - 32 * x01)),
                                     P[4 * mi + 2]);
                P[4 * mi + 3] = fmaf(s01.z, static_cast<float>(sc[1][0] * (d0[3] - 32 * x10) + sc[1][1] * (d1[3] - 32 * x11)),
                                     P[4 * mi + 3]);
            }
        }
        const float* dv = reinterpret_cast<const float*>(sl + kD) + (w >> 1) * kRows;
        const float dg0 = dv[g], dg1 = dv[g + 8];
#pragma unroll
        for (int mi = 0; mi < kN; ++mi) {
            acc[4 * mi + 0] = fmaf(dg0, P[4 * mi + 0], acc[4 * mi + 0]);
            acc[4 * mi + 1] = fmaf(dg0, P[4 * mi + 1], acc[4 * mi + 1]);
            acc[4 * mi + 2] = fmaf(dg1, P[4 * mi + 2], acc[4 * mi + 2]);
            acc[4 * mi + 3] = fmaf(dg1, P[4 * mi + 3], acc[4 * mi + 3]);
        }
    }
};

// Ring depth: as many stages as fit in 76 KB (at least 3).  With the staged
// activations that is just over a third of an SM's shared memory at m = 1, so
// two CTAs of a launch share an SM and a third cannot join them (measured:
// better than a 58 KB ring that lets three in, and than one or three CTAs
// per SM by grid size).  The 8- and 16-token forms stage 8-16 x more
// activations; there a 58 KB ring lets two CTAs share an SM for k = 4096
// (measured 10% faster at 8 tokens).
template <class F, int M>
__host__ __device__ constexpr int ring_depth() {
    return (M >= 8 ? 58 : 76) * 1024 / F::kSlot < 3 ? 3 : (M >= 8 ? 58 : 76) * 1024 / F::kSlot;
}

// ------------------------------------------------------------- layout --
struct StreamSmem {   // byte offsets: q8 [kc][M][32], (d_a, second term) fp32 [kc][M], row partial sums, ring
    size_t act, xs, red, ring, total;
    __host__ __device__ static size_t a16(size_t v) { return (v + 15) / 16 * 16; }
    __host__ __device__ StreamSmem(int mslots, int k, int depth, size_t slot) {
        const size_t kc = static_cast<size_t>(k) / 32;
        act = 0;
        xs = a16(static_cast<size_t>(mslots) * k);
        red = xs + a16(static_cast<size_t>(mslots) * kc * 8);
        ring = red + a16(static_cast<size_t>(kThreads / 32) * mslots * kRows * 4);
        total = ring + static_cast<size_t>(depth) * slot;
    }
};

// Bytes 0..7 of an 8-k group (words lo = k0..k3, hi = k4..k7) reordered to
// k = 0,4,1,5 | 2,6,3,7, the order of the nibble masks above.
__device__ __forceinline__ void permute_group(uint32_t lo, uint32_t hi, uint32_t& p0, uint32_t& p1) {
    const uint32_t a = __byte_perm(lo, hi, 0x5140), b = __byte_perm(lo, hi, 0x7362);
    p0 = a;
    p1 = b;
}

// Stage the m x k activations: the q8 SoA copied, or fp32 rows quantized by
// the q8 rule (a 32-element block per pair of threads); with each block's d_a
// and either d_a * ssum as fp32 (Q4_K) or the code sums of its two 16-element
// halves as two int16 in the bits of the second float (Q6_K).  Chunk-major
// (act [kc][M][32 B], xs [kc][M]): the tensor-core form's 8 tokens of a chunk
// are 256 contiguous bytes (8-byte loads without bank conflicts) and a token
// pair's scales one 16-byte load.
template <int M, bool kQuant, bool kPermuted, bool kHalfSums>
__device__ __forceinline__ void stage_acts(const GemvParams& p, int8_t* act, float2* xs) {
    const int kc = p.kc, m = p.m, k = p.k;
    if constexpr (kQuant) {
        // two adjacent threads per 32-element block, 16 elements each; every
        // lane takes part in each round (the shuffles), past the end idle
        const int halves = 2 * m * kc;
        for (int i0 = 0; i0 < halves; i0 += kThreads) {
            const int i = i0 + threadIdx.x;
            const bool live = i < halves;
            const int blk = live ? i >> 1 : 0, half = i & 1;
            const int t = blk / kc, c = blk - t * kc;
            const float4* src = reinterpret_cast<const float4*>(p.xf + static_cast<int64_t>(t) * p.ldx + 32 * c) + 4 * half;
            float v[16];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 f = live ? __ldg(src + e) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                v[4 * e] = f.x;
                v[4 * e + 1] = f.y;
                v[4 * e + 2] = f.z;
                v[4 * e + 3] = f.w;
            }
            float amax = fabsf(v[0]);
#pragma unroll
            for (int e = 1; e < 16; ++e) amax = fmaxf(amax, fabsf(v[e]));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            const Q8Scale s = q8_scale(amax);
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            int own = 0;   // this half's sum of codes
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int q = q8_code(v[e], s);
                own += q;
                w[e >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (e & 3));
            }
            const int sum = own + __shfl_xor_sync(0xFFFFFFFFu, own, 1);
            if constexpr (kPermuted) {
                permute_group(w[0], w[1], w[0], w[1]);
                permute_group(w[2], w[3], w[2], w[3]);
            }
            if (live) {
                reinterpret_cast<uint4*>(act + (static_cast<int64_t>(c) * M + t) * 32)[half] = make_uint4(w[0], w[1], w[2], w[3]);
                const float da = __half2float(s.da);
                if constexpr (kHalfSums) {
                    reinterpret_cast<int16_t*>(&xs[c * M + t].y)[half] = static_cast<int16_t>(own);
                    if (half == 0) xs[c * M + t].x = da;
                } else if (half == 0) {
                    xs[c * M + t] = make_float2(da, da * static_cast<float>(sum));
                }
            }
        }
    } else {
        const int v16 = k / 16;   // 16-B pieces of a q8 row
        for (int i = threadIdx.x; i < m * v16; i += kThreads) {
            const int t = i / v16, j = i - t * v16;
            uint4 w = __ldg(reinterpret_cast<const uint4*>(p.q8 + t * p.ldq) + j);
            if constexpr (kHalfSums) {   // piece j is half j % 2 of chunk j / 2
                const int hs = __dp4a(static_cast<int>(w.x), 0x01010101, __dp4a(static_cast<int>(w.y), 0x01010101,
                               __dp4a(static_cast<int>(w.z), 0x01010101, __dp4a(static_cast<int>(w.w), 0x01010101, 0))));
                reinterpret_cast<int16_t*>(&xs[(j >> 1) * M + t].y)[j & 1] = static_cast<int16_t>(hs);
            }
            if constexpr (kPermuted) {
                permute_group(w.x, w.y, w.x, w.y);
                permute_group(w.z, w.w, w.z, w.w);
            }
            reinterpret_cast<uint4*>(act + (static_cast<int64_t>(j >> 1) * M + t) * 32)[j & 1] = w;
        }
        for (int i = threadIdx.x; i < m * kc; i += kThreads) {
            const int t = i / kc, c = i - t * kc;
            const float da = __half2float(__ushort_as_half(__ldg(p.da + t * kc + c)));
            if constexpr (kHalfSums) {
                xs[c * M + t].x = da;
            } else {
                const float ss = static_cast<float>(__ldg(p.ssum + t * kc + c));
                xs[c * M + t] = make_float2(da, da * ss);
            }
        }
    }
}

template <class F, int M, bool kQuant>
__global__ void __launch_bounds__(kThreads, 2) gemv_stream_kernel(const GemvParams p) {
    constexpr int R = ring_depth<F, M>();
    constexpr int kSb = F::kStageSb;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const StreamSmem L(M, p.k, R, F::kSlot);
    int8_t* act = reinterpret_cast<int8_t*>(smem_raw + L.act);
    const float2* xs = reinterpret_cast<const float2*>(smem_raw + L.xs);
    float* red = reinterpret_cast<float*>(smem_raw + L.red);
    const uint32_t ring = smem_u32(smem_raw + L.ring);
    const int kc = p.kc, ksb = p.ksb, m = p.m, k = p.k;
    const int groups = p.n / kRows;
    // this CTA's groups: blockIdx.x, + G, + 2G, ... (the CTAs of one pass
    // read the 16-row slices of the same 128-row records at the same time)
    const int G = gridDim.x;
    const int g0 = blockIdx.x;
    const int mine = (groups - g0 + G - 1) / G;
    const int spg = (ksb + kSb - 1) / kSb;   // stages per group
    const int nst = mine * spg;

    // the next launch may start now; L2 is asked for this CTA's slice of the
    // weights (a hint; the copies below read after the wait)
    griddep_launch_dependents();
    if (threadIdx.x < 32) F::prefetch(p, blockIdx.x, gridDim.x);
    griddep_wait();

    // the stage the copies are issued for: group ig, super-blocks from isb
    typename F::Copier pc;
    pc.init();
    int ig = g0, isb = 0, islot = 0, issued = 0;
    if (nst > 0) pc.group(p, (static_cast<int64_t>(ig) * kRows) >> 7, (ig * kRows) & 127);
    auto issue = [&]() {   // the next stage into its ring slot (a commit group even when there is none)
        if (issued < nst) {
            pc.issue(ring + islot * F::kSlot, min(kSb, ksb - isb));
            ++issued;
            islot = islot + 1 == R ? 0 : islot + 1;
            isb += kSb;
            if (isb >= ksb) {
                isb = 0;
                ig += G;
                if (ig < groups) pc.group(p, (static_cast<int64_t>(ig) * kRows) >> 7, (ig * kRows) & 127);
            }
        }
        cp_async_commit();
    };
#pragma unroll 1
    for (int s = 0; s < R - 1; ++s) issue();
    stage_acts<M, kQuant, F::kPermuted, F::kHalfSums>(p, act, reinterpret_cast<float2*>(smem_raw + L.xs));

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = threadIdx.x & 15;
    const int j0 = (threadIdx.x >> 4) * F::kItems;   // this thread's first chunk in a stage
    constexpr bool kMma = M >= 8;                     // tensor-core form: warp w takes F::kMmaChunks chunks of a stage
    constexpr int kAcc = kMma ? M / 2 : M;
    float acc[kAcc];
#pragma unroll
    for (int t = 0; t < kAcc; ++t) acc[t] = 0.0f;
    int g = g0, sb0 = 0, slot = 0;   // the stage consumed
#pragma unroll 1
    for (int s = 0; s < nst; ++s) {
        cp_async_wait<R - 2>();   // this thread's copies of stage s have landed
        __syncthreads();          // everyone's have; everyone is done with stage s - 1 (and the activations are staged)
        issue();                  // into the slot stage s - 1 used
        const int nch = 8 * min(kSb, ksb - sb0);
        const uint8_t* sl = smem_raw + L.ring + static_cast<size_t>(slot) * F::kSlot;
        if constexpr (kMma) {
            if (F::kMmaChunks * warp < nch)
                F::template compute_mma<M>(sl, warp, lane, 8 * sb0 + F::kMmaChunks * warp, act, xs, k, kc, acc);
        } else {
            if (j0 < nch) F::template compute<M>(sl, j0, r, 8 * sb0 + j0, act, xs, m, k, kc, acc);
        }
        slot = slot + 1 == R ? 0 : slot + 1;
        sb0 += kSb;
        if (sb0 >= ksb) {   // the group's last stage: add the partial sums of each (token, row), store
            if constexpr (kMma) {   // each warp's (its super-blocks') sums, [warp][token][row]
                const int g = lane >> 2, q = lane & 3;
#pragma unroll
                for (int i = 0; i < kAcc; ++i) {
                    const int tok = 8 * (i >> 2) + 2 * q + (i & 1), row = g + 8 * ((i >> 1) & 1);
                    red[(warp * M + tok) * kRows + row] = acc[i];
                    acc[i] = 0.0f;
                }
            } else {   // the two half-warps of a row, then each warp's sums
#pragma unroll
                for (int t = 0; t < M; ++t) {
                    acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], 16);
                    if (lane < 16) red[(warp * M + t) * kRows + r] = acc[t];
                    acc[t] = 0.0f;
                }
            }
            __syncthreads();
            if (threadIdx.x < M * kRows) {
                const int t = threadIdx.x / kRows, rr = threadIdx.x % kRows;
                if (t < m) {
                    float v = 0.0f;
#pragma unroll
                    for (int w = 0; w < kThreads / 32; ++w) v += red[(w * M + t) * kRows + rr];
                    const int64_t o = static_cast<int64_t>(g) * kRows + rr;
                    if (p.out_bf16)
                        static_cast<__nv_bfloat16*>(p.y)[t * p.ldy + o] = __float2bfloat16_rn(v);
                    else
                        static_cast<float*>(p.y)[t * p.ldy + o] = v;
                }
            }
            sb0 = 0;
            g += G;
        }
    }
    cp_async_wait<0>();   // no copy outlives the CTA (the trailing groups are empty)
}

template <class F, int M, bool kQuant>
cudaError_t launch_stream_m(const GemvParams& p, cudaStream_t s, bool* launched) {
    *launched = false;
    const size_t smem = StreamSmem(M, p.k, ring_depth<F, M>(), F::kSlot).total;
    if (smem > kStreamMaxSmem) return cudaSuccess;   // too large: the caller uses another form
    static std::atomic<bool> attr_set[64];   // zero at start; a race only repeats the call
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(gemv_stream_kernel<F, M, kQuant>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kStreamMaxSmem));
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_stream_kernel<F, M, kQuant>, kThreads,
                                                          smem)) != cudaSuccess)
        return e;
    // two CTAs a SM where they fit (m <= 4), one with the larger staged activations of 8 or 16 tokens
    const int groups = static_cast<int>(p.n / kRows);
    const int grid = std::max(1, std::min(groups, std::min(2, std::max(1, per_sm)) * sms));
    *launched = true;
    return launch_pdl(gemv_stream_kernel<F, M, kQuant>, dim3(grid), dim3(kThreads), smem, s, p);
}

template <class F, bool kQuant>
cudaError_t launch_stream_any(const GemvParams& p, cudaStream_t s, bool* launched) {
    if (p.m <= 1) return launch_stream_m<F, 1, kQuant>(p, s, launched);
    if (p.m <= 2) return launch_stream_m<F, 2, kQuant>(p, s, launched);
    if (p.m <= 4) return launch_stream_m<F, 4, kQuant>(p, s, launched);
    if constexpr (F::kMma && !kQuant) {   // 5..16 tokens, q8 input: the tensor-core form
        if (p.m <= 8) return launch_stream_m<F, 8, false>(p, s, launched);
        cudaError_t e = launch_stream_m<F, 16, false>(p, s, launched);
        if (e != cudaSuccess || *launched) return e;
        // 16 tokens of a long k do not fit: tokens 0-7, then the rest, each a
        // pass over the weights (measured: faster than the register-held kernel)
        GemvParams lo = p, hi = p;
        lo.m = 8;
        hi.m = p.m - 8;
        hi.q8 = p.q8 + 8 * p.ldq;
        hi.da = p.da + 8 * static_cast<int64_t>(p.kc);
        hi.ssum = p.ssum + 8 * static_cast<int64_t>(p.kc);
        hi.y = p.out_bf16 ? static_cast<void*>(static_cast<__nv_bfloat16*>(p.y) + 8 * p.ldy)
                          : static_cast<void*>(static_cast<float*>(p.y) + 8 * p.ldy);
        if ((e = launch_stream_m<F, 8, false>(lo, s, launched)) != cudaSuccess || !*launched) return e;
        return launch_stream_m<F, 8, false>(hi, s, launched);
    }
    return cudaSuccess;   // not this kernel's range: *launched stays false
}

}  // namespace

cudaError_t launch_gemv_stream(const GemvParams& p, cudaStream_t s, bool* launched) {
    *launched = false;
    if (p.m < 1 || p.m > 16 || p.n % kRows) return cudaSuccess;
    if (p.q6) return p.xf ? launch_stream_any<Q6Stream, true>(p, s, launched)
                          : launch_stream_any<Q6Stream, false>(p, s, launched);
    return p.xf ? launch_stream_any<Q4Stream, true>(p, s, launched)
                : launch_stream_any<Q4Stream, false>(p, s, launched);
}

}  // namespace q4k

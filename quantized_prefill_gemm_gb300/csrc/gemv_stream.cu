// Small-M (decode-sized) product with the packed weights streamed through a
// shared-memory ring: m <= 4 tokens, Q4_K or Q6_K weights.
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
//   - two CTAs of 256 threads per SM (grid G = min(row groups, 2 x SMs)); CTA b
//     owns the 16-row groups b, b + G, b + 2G, ..., every group over all of
//     k, so no partial sum leaves the CTA, and the CTAs working at the same
//     time read neighbouring slices of the same 128-row records;
//   - the CTA's weights flow through a ring of R stages (a few super-blocks
//     of one group each) filled with 16-byte cp.async copies, R-1 stages in
//     flight while one is consumed; their completion is the hardware's
//     wait_group, so no thread spins on a flag;
//   - a CTA takes under a third of an SM (256 threads, about 70 KB of shared
//     memory), so a CTA of the next launch is resident while this one runs.  Launched with programmatic dependent launch, each asks L2 for a
//     1/G slice of its launch's weights (a prefetch hint: it cannot change
//     what a later load returns) and only then waits for the kernel before
//     it, so the weights come from HBM while that kernel finishes.  Every
//     read of the ring or of the activations comes after the wait.
//
// Q4_K without unpacking: in a packed quant word the nibbles of k = 0,4,1,5
// sit at bits 0, 8, 16, 24 and those of k = 2,6,3,7 at bits 4, 12, 20, 28
// (the word layout of the packed format), so w & 0x0F0F0F0F and
// (w >> 4) & 0x0F0F0F0F are byte vectors dp4a takes as they are, against the
// activations staged with each 8-byte group reordered to k = 0,4,1,5,2,6,3,7.
// The integer dot product is the same sum in another order.
//
// Thread t takes row r = t % 16 of the group and the stage's chunks
// (t / 16) * I .. + I - 1 (I = 4 for Q4_K, 2 for Q6_K; one super-block); a
// row's sums are added over its 16 threads (a shuffle, then 8 warps' partials
// in shared memory in a fixed order) at the end of each group and stored.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <algorithm>

#include "q4k_internal.h"
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
// b + 2G, ... (over the grid, the whole array; no division on the way).
__device__ __forceinline__ void prefetch_pages(const void* base, int64_t bytes, int b, int G) {
    const int64_t pages = (bytes + 4095) >> 12;
    for (int64_t pg = b + static_cast<int64_t>(G) * threadIdx.x; pg < pages; pg += static_cast<int64_t>(G) * kThreads) {
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

// Q4_K: nib 16 B, sc 1 B, m 1 B per (row, chunk); d, dmin fp32 per (row, sb).
// A stage is 8 super-blocks; a thread takes 4 chunks of one super-block.
struct Q4Stream {
    static constexpr int kStageSb = 8;
    static constexpr int kItems = 4;
    static constexpr bool kPermuted = true;   // activations staged in the nibble order
    static constexpr int kArrays = 5;         // nib, sc, m, d, dmin
    static constexpr uint32_t kNib = 0;
    static constexpr uint32_t kSc = kNib + 8 * kStageSb * kRows * 16;
    static constexpr uint32_t kMq = kSc + 8 * kStageSb * kRows;
    static constexpr uint32_t kD = kMq + 8 * kStageSb * kRows;
    static constexpr uint32_t kDmin = kD + kStageSb * kRows * 4;
    static constexpr uint32_t kSlot = kDmin + kStageSb * kRows * 4;
    __host__ __device__ static constexpr int bpr(int a) { return a == 0 ? 16 : a < 3 ? 1 : 4; }
    __host__ __device__ static constexpr bool per_sb(int a) { return a >= 3; }
    __host__ __device__ static constexpr uint32_t smem_off(int a) {
        return a == 0 ? kNib : a == 1 ? kSc : a == 2 ? kMq : a == 3 ? kD : kDmin;
    }
    __device__ static const void* base(const GemvParams& p, int a) {
        return a == 0 ? static_cast<const void*>(p.nib) : a == 1 ? static_cast<const void*>(p.sc)
             : a == 2 ? static_cast<const void*>(p.mq) : a == 3 ? static_cast<const void*>(p.dsb)
                      : static_cast<const void*>(p.dmn);
    }
    __device__ static void prefetch(const GemvParams& p, int b, int G) {
        const int64_t n = p.n;
        prefetch_pages(p.nib, n * p.k / 2, b, G);
        prefetch_pages(p.sc, n * p.kc, b, G);
        prefetch_pages(p.mq, n * p.kc, b, G);
        prefetch_pages(p.dsb, n * p.ksb * 4, b, G);
        prefetch_pages(p.dmn, n * p.ksb * 4, b, G);
    }
    // Row r, chunks j0 .. j0 + 3 of the stage (global chunks c0 .. c0 + 3):
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
                    const int4* a = reinterpret_cast<const int4*>(act + static_cast<int64_t>(t) * k + 32 * c);
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
                    const float2 s = xs[t * kc + c];   // d_a, d_a * ssum (both exact in fp32)
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
};

// Q6_K: lo 16 B, hi 8 B, the two i8 scales 2 B per (row, chunk); d fp32 per
// (row, sb).  A stage is 4 super-blocks; a thread takes 2 chunks of one.
struct Q6Stream {
    static constexpr int kStageSb = 4;
    static constexpr int kItems = 2;
    static constexpr bool kPermuted = false;
    static constexpr uint32_t kLo = 0;
    static constexpr uint32_t kHi = kLo + 8 * kStageSb * kRows * 16;
    static constexpr uint32_t kSc = kHi + 8 * kStageSb * kRows * 8;
    static constexpr uint32_t kD = kSc + 8 * kStageSb * kRows * 2;
    static constexpr uint32_t kSlot = kD + kStageSb * kRows * 4;

    static constexpr int kArrays = 4;         // lo, hi, the scale pair, d
    __host__ __device__ static constexpr int bpr(int a) { return a == 0 ? 16 : a == 1 ? 8 : a == 2 ? 2 : 4; }
    __host__ __device__ static constexpr bool per_sb(int a) { return a == 3; }
    __host__ __device__ static constexpr uint32_t smem_off(int a) {
        return a == 0 ? kLo : a == 1 ? kHi : a == 2 ? kSc : kD;
    }
    __device__ static const void* base(const GemvParams& p, int a) {
        return a == 0 ? static_cast<const void*>(p.nib) : a == 1 ? static_cast<const void*>(p.q6hi)
             : a == 2 ? static_cast<const void*>(p.sc) : static_cast<const void*>(p.dsb);
    }
    __device__ static void prefetch(const GemvParams& p, int b, int G) {
        const int64_t n = p.n;
        prefetch_pages(p.nib, n * p.k / 2, b, G);
        prefetch_pages(p.q6hi, n * p.k / 4, b, G);
        prefetch_pages(p.sc, n * p.kc * 2, b, G);
        prefetch_pages(p.dsb, n * p.ksb * 4, b, G);
    }
    // I = sc_0 * sum_{k<16} (q-32) qa + sc_1 * sum_{k>=16} (q-32) qa (|I| < 2^24, exact in fp32)
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
            uint32_t v[8];
            unpack_q6(lo.x, hi.x, v[0], v[1]);
            unpack_q6(lo.y, hi.x >> 2, v[2], v[3]);
            unpack_q6(lo.z, hi.y, v[4], v[5]);
            unpack_q6(lo.w, hi.y >> 2, v[6], v[7]);
            const int sc0 = static_cast<int>(static_cast<int8_t>(scp & 0xFFu));
            const int sc1 = static_cast<int>(static_cast<int8_t>(scp >> 8));
#pragma unroll
            for (int t = 0; t < M; ++t) {
                if (t < m) {
                    const int4* a = reinterpret_cast<const int4*>(act + static_cast<int64_t>(t) * k + 32 * c);
                    const int4 a0 = a[0], a1 = a[1];
                    int J0 = __dp4a(static_cast<int>(v[0]), a0.x, 0);
                    J0 = __dp4a(static_cast<int>(v[1]), a0.y, J0);
                    J0 = __dp4a(static_cast<int>(v[2]), a0.z, J0);
                    J0 = __dp4a(static_cast<int>(v[3]), a0.w, J0);
                    int J1 = __dp4a(static_cast<int>(v[4]), a1.x, 0);
                    J1 = __dp4a(static_cast<int>(v[5]), a1.y, J1);
                    J1 = __dp4a(static_cast<int>(v[6]), a1.z, J1);
                    J1 = __dp4a(static_cast<int>(v[7]), a1.w, J1);
                    P[t] = fmaf(xs[t * kc + c].x, static_cast<float>(sc0 * J0 + sc1 * J1), P[t]);
                }
            }
        }
        const float d = reinterpret_cast<const float*>(sl + kD)[(j0 >> 3) * kRows + r];
#pragma unroll
        for (int t = 0; t < M; ++t) acc[t] = fmaf(d, P[t], acc[t]);
    }
};

// The 16-byte pieces this thread copies for every stage.  A full stage's
// pieces are numbered array by array (each array's records in order, kBpr
// pieces a record) and piece i is copied by thread i % 256; what a thread
// owns is worked out once, and per stage only its source pointers move on.
template <class F>
__host__ __device__ constexpr int stage_pieces() {
    int n = 0;
    for (int a = 0; a < F::kArrays; ++a) n += (F::per_sb(a) ? 1 : 8) * F::kStageSb * F::bpr(a);
    return n;
}

template <class F>
struct Pieces {
    static constexpr int kPer = (stage_pieces<F>() + kThreads - 1) / kThreads;
    const uint8_t* src[kPer];   // the piece of the next stage issued
    uint32_t dst[kPer];         // its offset in a ring slot
    int arr[kPer];              // its array, -1 for none
    int off[kPer];              // its offset from the array's first record (row r0) of a stage
    int usb[kPer];              // its super-block within a stage (copied while usb < the stage's super-blocks)
    int step[kPer];             // bytes from one stage's piece to the next one's

    __device__ void init() {
#pragma unroll
        for (int h = 0; h < kPer; ++h) {
            int i = threadIdx.x + kThreads * h;
            arr[h] = -1;
            dst[h] = 0;
            off[h] = 0;
            usb[h] = 0;
            step[h] = 0;
            src[h] = nullptr;
#pragma unroll
            for (int a = 0; a < F::kArrays; ++a) {
                const int n = (F::per_sb(a) ? 1 : 8) * F::kStageSb * F::bpr(a);
                if (arr[h] < 0 && i < n) {
                    const int u = i / F::bpr(a), part = i % F::bpr(a);
                    arr[h] = a;
                    dst[h] = F::smem_off(a) + 16 * i;
                    off[h] = u * 128 * F::bpr(a) + 16 * part;
                    usb[h] = F::per_sb(a) ? u : u >> 3;
                    step[h] = (F::per_sb(a) ? 1 : 8) * F::kStageSb * 128 * F::bpr(a);
                }
                if (arr[h] < 0) i -= n;
            }
        }
    }
    // first stage of the 16-row group at rows row0 (tile nt, row r0 in it)
    __device__ void group(const GemvParams& p, int64_t nt, int r0) {
#pragma unroll
        for (int h = 0; h < kPer; ++h) {
#pragma unroll
            for (int a = 0; a < F::kArrays; ++a) {
                if (arr[h] == a) {
                    const int64_t rec = F::per_sb(a) ? nt * p.ksb : nt * p.kc;
                    src[h] = static_cast<const uint8_t*>(F::base(p, a)) + (rec * 128 + r0) * F::bpr(a) + off[h];
                }
            }
        }
    }
    // copy the stage of ns super-blocks into the slot at smem address slot, then step to the next stage
    __device__ void issue(uint32_t slot, int ns) {
#pragma unroll
        for (int h = 0; h < kPer; ++h) {
            if (arr[h] >= 0 && usb[h] < ns) cp_async16(slot + dst[h], src[h]);
            src[h] += step[h];
        }
    }
};

// Ring depth: as many stages as fit in 58 KB (at least 3), so that two CTAs of
// this launch and one of the next share an SM for k up to 11008 at m = 1
// (measured: two CTAs of a launch per SM beat one or three).
template <class F, int M>
__host__ __device__ constexpr int ring_depth() {
    return 58 * 1024 / F::kSlot < 3 ? 3 : 58 * 1024 / F::kSlot;
}

// ------------------------------------------------------------- layout --
struct StreamSmem {   // byte offsets: q8 [m][k], (d_a, d_a*ssum) fp32 [m][kc], row partial sums, ring
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
// and d_a * ssum as fp32.
template <bool kQuant, bool kPermuted>
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
            int sum = 0;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int q = q8_code(v[e], s);
                sum += q;
                w[e >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (e & 3));
            }
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
            if constexpr (kPermuted) {
                permute_group(w[0], w[1], w[0], w[1]);
                permute_group(w[2], w[3], w[2], w[3]);
            }
            if (live) {
                reinterpret_cast<uint4*>(act + static_cast<int64_t>(t) * k + 32 * c)[half] = make_uint4(w[0], w[1], w[2], w[3]);
                if (half == 0) {
                    const float da = __half2float(s.da);
                    xs[t * kc + c] = make_float2(da, da * static_cast<float>(sum));
                }
            }
        }
    } else {
        const int v16 = k / 16;   // 16-B pieces of a q8 row
        for (int i = threadIdx.x; i < m * v16; i += kThreads) {
            const int t = i / v16, j = i - t * v16;
            uint4 w = __ldg(reinterpret_cast<const uint4*>(p.q8 + t * p.ldq) + j);
            if constexpr (kPermuted) {
                permute_group(w.x, w.y, w.x, w.y);
                permute_group(w.z, w.w, w.z, w.w);
            }
            reinterpret_cast<uint4*>(act + static_cast<int64_t>(t) * k)[j] = w;
        }
        for (int i = threadIdx.x; i < m * kc; i += kThreads) {
            const int t = i / kc, c = i - t * kc;
            const float da = __half2float(__ushort_as_half(__ldg(p.da + t * kc + c)));
            const float ss = p.ssum ? static_cast<float>(__ldg(p.ssum + t * kc + c)) : 0.0f;
            xs[t * kc + c] = make_float2(da, da * ss);
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
    F::prefetch(p, blockIdx.x, gridDim.x);
    griddep_wait();

    // the stage the copies are issued for: group ig, super-blocks from isb
    Pieces<F> pc;
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
    stage_acts<kQuant, F::kPermuted>(p, act, reinterpret_cast<float2*>(smem_raw + L.xs));

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = threadIdx.x & 15;
    const int j0 = (threadIdx.x >> 4) * F::kItems;   // this thread's first chunk in a stage
    float acc[M];
#pragma unroll
    for (int t = 0; t < M; ++t) acc[t] = 0.0f;
    int g = g0, sb0 = 0, slot = 0;   // the stage consumed
#pragma unroll 1
    for (int s = 0; s < nst; ++s) {
        cp_async_wait<R - 2>();   // this thread's copies of stage s have landed
        __syncthreads();          // everyone's have; everyone is done with stage s - 1 (and the activations are staged)
        issue();                  // into the slot stage s - 1 used
        const int nch = 8 * min(kSb, ksb - sb0);
        if (j0 < nch)
            F::template compute<M>(smem_raw + L.ring + static_cast<size_t>(slot) * F::kSlot, j0, r, 8 * sb0 + j0, act,
                                   xs, m, k, kc, acc);
        slot = slot + 1 == R ? 0 : slot + 1;
        sb0 += kSb;
        if (sb0 >= ksb) {   // the group's last stage: add the 32 threads of each row, store
#pragma unroll
            for (int t = 0; t < M; ++t) {
                acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], 16);
                if (lane < 16) red[(warp * M + t) * kRows + r] = acc[t];
                acc[t] = 0.0f;
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
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(gemv_stream_kernel<F, M, kQuant>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kStreamMaxSmem));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int groups = static_cast<int>(p.n / kRows);
    const int grid = std::max(1, std::min(groups, 2 * sms));   // two CTAs a SM
    *launched = true;
    return launch_pdl(gemv_stream_kernel<F, M, kQuant>, dim3(grid), dim3(kThreads), smem, s, p);
}

template <class F, bool kQuant>
cudaError_t launch_stream_any(const GemvParams& p, cudaStream_t s, bool* launched) {
    if (p.m <= 1) return launch_stream_m<F, 1, kQuant>(p, s, launched);
    if (p.m <= 2) return launch_stream_m<F, 2, kQuant>(p, s, launched);
    return launch_stream_m<F, 4, kQuant>(p, s, launched);
}

}  // namespace

cudaError_t launch_gemv_stream(const GemvParams& p, cudaStream_t s, bool* launched) {
    *launched = false;
    if (p.m < 1 || p.m > 4 || p.n % kRows) return cudaSuccess;
    if (p.q6) return p.xf ? launch_stream_any<Q6Stream, true>(p, s, launched)
                          : launch_stream_any<Q6Stream, false>(p, s, launched);
    return p.xf ? launch_stream_any<Q4Stream, true>(p, s, launched)
                : launch_stream_any<Q4Stream, false>(p, s, launched);
}

}  // namespace q4k

// Q4_K x q8 prefill GEMM on sm_103a tensor cores.
//
//   Y[t, o] = sum_sb d[o,sb] * sum_{c in sb} da[t,c] * J_c[t,o]  -  Z[t,o]
//   J_c[t,o] = sum_{k in c} (sc*q)[o,k] * qa[t,k]          (exact integer)
//   Z[t,o]   = sum_c (da*ssum)[t,c] * (dmin*m)[o,c]        (min term)
//
// This is the per-32-k integer dot product plus the two-term rank-1 rescale
// of "34 · r31 — q-major sda scale-read repack" (§1: A-side d and ssum per
// token and chunk; §2: B-side d*sc and -dmin*m per chunk and od row) and the
// r15 rank-1 fold named in "22 · r17 — Wide warp remap" (§1), regrouped:
// d*sc*I splits into sc*I (folded into the weight operand) and d (applied
// once per super-block), and the -dmin*m*ssum*da term, a rank-1 product per
// chunk, becomes one small GEMM of depth k/32.
//
// sm_103a has no integer tcgen05 MMA, so the integer dot products run on the
// f16 kind: qa in [-127, 127] and sc*q in [0, 945] are exact fp16 integers,
// every product is exact, and a 32-term chunk sum stays below 2^22, so the
// fp32 TMEM accumulator holds J_c exactly.  The min-term GEMM runs in bf16 on
// hi/lo splits of both operands (three MMAs: hi*hi + hi*lo + lo*hi, relative
// error ~2^-16 per term, far inside the 1e-4 * sum|w*a| bound).
//
// One persistent CTA per SM (512 threads, 16 warps), one 128-token x 128-od
// output tile at a time, k in stages of 128 for Q4_K and 64 for Q6_K (four or
// two chunks of 32):
//   warp 0        TMA producer: activation tile (fp16, 128-B swizzle), packed
//                 quants and sc; d at super-block ends, into a ring of its
//                 own; for the min-term stages the bf16 E and -(dmin*m) tiles
//   warp 1        MMA issuer: 2 x (M128 N128 K16) per chunk, two chunks into
//                 the two accumulators of one TMEM group, one commit for both;
//                 12 bf16 MMAs per 64 of min-term depth (hi*hi, hi*lo, lo*hi)
//                 into a group's first one
//   warps 2-3     no role (they complete the first warpgroup); with the
//                 in-kernel quantization (kQuant) they quantize the
//                 activation items the first wave of tiles does not need
//   warps 4-7     converters: 4-bit quants -> fp16 sc*q written in the
//                 128-B-swizzled K-major layout the MMA reads
//   warps 8-15    drain: per chunk, P += da * J (packed fp32 FMA) from TMEM;
//                 per super-block Y += d * P; per tile Y -> HBM.  Y and P live
//                 in registers (setmaxnreg gives these warps 184 each).  With
//                 kQuant they first quantize the first wave's items.
// TMEM (512 columns): two groups of two 128-column accumulators.  A group is
// handed over once per two chunks, which halves the MMA <-> drain hand-offs
// of a per-chunk scheme; those hand-offs, not the tensor pipe, bound the loop.
// Every wait is bounded (q4k_ptx.cuh: mbar_wait): a stuck pipeline records an
// error word and the CTA leaves through the normal teardown.
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4k_internal.h"
#include "q4k_layout.h"
#include "q4k_ptx.cuh"
#include "q4k_unpack.cuh"
#include "q8_operand.cuh"
#include "q8_rule.cuh"

namespace q4k {
namespace {

constexpr int kThreads = 512;

// Shared-memory carve-out per format.  Q4_K: three stages of 128 k (four
// 32-k chunks) holding the fp16 A tile, the fp16 B tile (sc*q), the packed
// quants and sc.  Q6_K: four stages of 64 k (the B tile has two fp16
// planes, the sh and the sl part of the scale) plus the high quant bits.  A and B tiles are made of
// 16 KB boxes of 128 rows x 64 k (128-B rows, 128-B swizzle), one per two
// chunks.  A min-term stage holds 64 of depth: the hi and the lo box of E in
// the A slots, those of -(dmin*m) in the B slots (Q4_K only).
// The super-block scales d have a ring of their own, shared by the producer
// and the drain only, so that the drain (the slowest role) never holds a
// stage of the main ring.
template <bool kQ6>
struct Lay {
    static constexpr int kCh = gemm_chunks_per_stage(kQ6);     // 32-k chunks per main stage
    static constexpr int kStPerSb = 8 / kCh;                    // main stages per super-block
    static constexpr int kStages = kQ6 ? 4 : 3;
    static constexpr uint32_t kBox = 16384;                     // 128 rows x 64 fp16 / bf16
    static constexpr uint32_t kStageA = kBox * (kCh / 2);
    static constexpr uint32_t kStageB = kQ6 ? 2 * kBox : kBox * (kCh / 2);   // Q6_K: sh plane, then sl plane
    static constexpr uint32_t kStageNib = 2048 * kCh;           // chunks x 128 rows x 16 B
    static constexpr uint32_t kStageHi = kQ6 ? 1024 * kCh : 0;  // chunks x 128 rows x 8 B
    static constexpr uint32_t kStageSc = (kQ6 ? 256 : 128) * kCh;   // chunks x 128 rows x (2 or 1) B
    static constexpr uint32_t kSlotD = 512;                     // 128 rows x fp32, one super-block
    static constexpr int kDRing = 4;                            // d slots (super-blocks in flight)
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kOffA + kStages * kStageA;
    static constexpr uint32_t kOffNib = kOffB + kStages * kStageB;
    static constexpr uint32_t kOffHi = kOffNib + kStages * kStageNib;
    static constexpr uint32_t kOffSc = kOffHi + kStages * kStageHi;
    static constexpr uint32_t kOffD = kOffSc + kStages * kStageSc;
    static constexpr uint32_t kOffBar = kOffD + kDRing * kSlotD;
    // barrier indices
    static constexpr int kBarFull = 0;                       // [kStages] producer -> all (tx bytes)
    static constexpr int kBarConv = kStages;                 // [kStages] converters -> MMA (4 arrivals)
    static constexpr int kBarEmpty = 2 * kStages;            // [kStages] MMA commit -> producer
    static constexpr int kBarAccFull = 3 * kStages;          // [2] MMA commit -> drain (one accumulator group)
    static constexpr int kBarAccEmpty = kBarAccFull + 2;     // [2] 8 drain warps -> MMA
    static constexpr int kBarDrain = kBarAccEmpty + 2;       // MMA's final commit
    static constexpr int kBarDFull = kBarDrain + 1;          // [kDRing] producer -> drain (tx bytes)
    static constexpr int kBarDEmpty = kBarDFull + kDRing;    // [kDRing] 8 drain warps -> producer
    static constexpr int kNumBars = kBarDEmpty + kDRing;
    static constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;   // TMEM base slot, abort flag, ready unit
    static constexpr uint32_t kSmemUsed = kOffMisc + 16;
    static constexpr size_t kSmemBytes = kSmemUsed + 1024;          // + alignment slack
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Per-thread registers after the re-split (warpgroups 0, 1 and 2-3).  The
// launch gives every thread 65536 / 512 = 128; the shares must not add up to
// more than that total, or the increase would wait forever.
constexpr uint32_t kRegsCtl = 56, kRegsConv = 80, kRegsDrain = 184;
static_assert(128 * kRegsCtl + 128 * kRegsConv + 256 * kRegsDrain <= 65536, "register re-split exceeds the launch");

constexpr uint32_t kIdescMain = idesc_kind_f16(128, 128, false);   // fp16 x fp16 -> fp32
constexpr uint32_t kIdescMin = idesc_kind_f16(128, 128, true);     // bf16 x bf16 -> fp32

// wait sites recorded in the error word (numbers kept stable; 2 is no longer
// used: the running Y left TMEM, and with it the MMA's wait for a free Y)
enum : unsigned {
    kSiteProdEmpty = 1, kSiteUnused2, kSiteMmaFull, kSiteMmaConv, kSiteMmaAccEmpty,
    kSiteConvFull, kSiteEpiD, kSiteEpiAccFull, kSiteEpiZ, kSiteProdD,
    kSiteProdQuant, kSiteEpiReady, kSiteQuantArrive
};

template <bool kQ6>
struct Ctx {
    using L = Lay<kQ6>;
    uint32_t base;      // shared address of the 1024-aligned carve-out
    uint8_t* sbase;     // generic pointer to the same
    uint32_t tmem;      // TMEM base address (lane 0, column 0)
    volatile int* abort_flag;
    uint32_t ready;     // shared address of the ready-unit word (in-kernel quantization)
    __device__ uint32_t bar(int i) const { return base + L::kOffBar + 8u * static_cast<uint32_t>(i); }
    __device__ uint32_t a(int s) const { return base + L::kOffA + L::kStageA * s; }
    __device__ uint32_t b(int s) const { return base + L::kOffB + L::kStageB * s; }
    __device__ bool wait(const GemmParams& p, int barrier, uint32_t parity, unsigned site) const {
        return mbar_wait(bar(barrier), parity, abort_flag, p.timeout_cycles, p.err, site);
    }
    // all 32 lanes wait; the warp proceeds only if every lane saw the phase
    __device__ bool warp_wait(const GemmParams& p, int barrier, uint32_t parity, unsigned site) const {
        const bool ok = wait(p, barrier, parity, site);
        return __all_sync(0xFFFFFFFFu, ok);
    }
};

template <bool kQ6>
__device__ __forceinline__ void advance(int& s, uint32_t& ph) {
    if (++s == Lay<kQ6>::kStages) {
        s = 0;
        ph ^= 1u;
    }
}

template <bool kQ6>
__device__ __forceinline__ void advance_d(int& ds, uint32_t& dph) {
    if (++ds == Lay<kQ6>::kDRing) {
        ds = 0;
        dph ^= 1u;
    }
}

// One work unit: a whole tile, or one k-part of a tail tile (GemmParams).
// Its stages st = 0 .. n_st-1 map to kb = st + kbase: kb < 0 are the
// min-term stages (a unit has all of them or none: only whole tiles and part
// 0 have them, and those start at kb = 0), kb >= 0 the main stages of kCh
// chunks.
struct Unit {
    int mt, nt;
    int kbase;      // first main stage minus the number of min-term stages
    int n_st;       // stages of this unit
    int slot;       // tail tile x split + part for a k-part, -1 for a whole tile
};

template <bool kQ6>
__device__ __forceinline__ Unit unit_of(const GemmParams& p, int u) {
    constexpr int kSps = Lay<kQ6>::kStPerSb;
    Unit w;
    int tile;
    if (u < p.full_tiles) {
        tile = u;
        w.slot = -1;
        w.kbase = -p.n_zst;
        w.n_st = p.n_zst + p.n_main;
    } else {
        const int v = u - p.full_tiles;
        const int tail = v / p.split, part = v - tail * p.split;
        tile = p.full_tiles + tail;
        w.slot = v;
        const int kb0 = kSps * part * p.part_sb, kb1 = min(p.n_main, kb0 + kSps * p.part_sb);
        const int zst = part == 0 ? p.n_zst : 0;
        w.kbase = kb0 - zst;
        w.n_st = zst + kb1 - kb0;
    }
    if (p.nt_fast) {
        w.nt = tile % p.n_tiles;
        w.mt = tile / p.n_tiles;
    } else {
        w.mt = tile % p.m_tiles;
        w.nt = tile / p.m_tiles;
    }
    return w;
}

// ------------------------------------------------ in-kernel quantization --
// With x given in fp32 the kernel writes the activation operand itself, with
// the routine of the separate pass (quantize_pair_block), so the bits are the
// same.  The work is cut into items, (token tile, slice of its kc blocks),
// qs slices a tile.  A CTA's items are done by warps that have nothing else
// to do at that moment: the items the first wave of tiles needs by the eight
// drain warps before their first accumulator, the rest by the two spare
// warps while the tiles run.  With the output tile fastest in the tile order
// the first wave needs only the first ceil(grid / n_tiles) token tiles.  A
// finished item adds one to its token tile's count, tagged with the call so
// that counts of an earlier call on the same workspace are never mistaken
// for this one's; the producer waits for a full count (qs items) before the
// first copy of a unit's activation tiles and tells the drain (which reads
// d_a with plain loads) through a ready word in shared memory.

// Item `it` with `nw` warps (this one is number qw): passes of 16 * kR
// (token, block) pairs a warp, each lane with the loads of kR pairs in flight.
template <int kR>
__device__ __forceinline__ void quantize_item(const GemmParams& p, int it, int nw, int qw, int lane) {
    const int mt = it / p.qs, j = it - mt * p.qs;
    const int c0 = static_cast<int>(static_cast<int64_t>(j) * p.kc / p.qs);
    const int nb = static_cast<int>(static_cast<int64_t>(j + 1) * p.kc / p.qs) - c0;
    const int pairs = 128 * nb;
    for (int base = 16 * kR * qw; base < pairs; base += 16 * kR * nw) {
        float v[kR][16];
        int64_t t[kR], c[kR];
        bool in[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) {
            const int q = base + 16 * r + (lane >> 1);
            in[r] = q < pairs;
            const int tt = in[r] ? q / nb : 0;
            t[r] = static_cast<int64_t>(mt) * 128 + tt;
            c[r] = c0 + (in[r] ? q - tt * nb : 0);
            pair_load(p.xf, p.ldx, p.m, t[r], c[r], lane & 1, in[r], v[r]);
        }
#pragma unroll
        for (int r = 0; r < kR; ++r)
            pair_finish(v[r], p.m, p.k, p.kc, t[r], c[r], lane & 1, in[r], p.xq_w, p.da_w, p.e_w);
    }
}

// One item of token tile mt finished (the caller has ordered every write of
// it before this thread, by a barrier): release it into the tile's count.  The
// first arrival of a call finds the word under another tag (an earlier call's,
// or whatever the workspace held) and installs this call's with a count of
// one; every other arrival adds one.  Only this call writes the word while it
// runs, so the exchange is retried at most once (after losing the
// installation to another arrival of this call); the additions queue in L2
// instead of retrying round trips.
__device__ __forceinline__ void quantize_arrive(const GemmParams& p, int mt) {
    fence_proxy_async_global();
    fence_acq_rel_gpu();
    unsigned long long* f = p.qflag + mt;
    unsigned long long cur = ld_relaxed_gpu_u64(f);
    for (int i = 0; i < 4; ++i) {
        if ((cur & ~0xFFFFull) == p.qtag) {
            atomicAdd(f, 1ull);
            return;
        }
        const unsigned long long prev = atomicCAS(f, cur, p.qtag | 1ull);
        if (prev == cur) return;
        cur = prev;
    }
    atomicCAS(p.err, 0u, kErrTimeoutBase | kSiteQuantArrive);
}

// Items it0, it0 + gridDim.x, ... below it_end with the nw warps that call
// this together (named barrier `bar`; warp number qw among them).
template <int kR>
__device__ __forceinline__ void quantize_items(const GemmParams& p, int it0, int it_end, int nw, int qw, int lane,
                                               uint32_t bar) {
    for (int it = it0; it < it_end; it += gridDim.x) {
        quantize_item<kR>(p, it, nw, qw, lane);
        fence_proxy_async_global();   // the writes, for the other CTAs' tensor copies
        named_bar_sync(bar, 32u * static_cast<uint32_t>(nw));
        if (qw == 0 && lane == 0) quantize_arrive(p, it / p.qs);
    }
}

// The producer's wait for a full count of token tile mt, then the acquire.
__device__ __forceinline__ bool quantize_wait(const GemmParams& p, int mt, volatile int* abort) {
    const unsigned long long want = p.qtag | static_cast<unsigned long long>(p.qs);
    const unsigned long long* f = p.qflag + mt;
    if (ld_relaxed_gpu_u64(f) != want) {
        const long long t0 = clock64();
        while (ld_relaxed_gpu_u64(f) != want) {
            __nanosleep(100);
            if (*abort) return false;
            if (static_cast<uint64_t>(clock64() - t0) > p.timeout_cycles) {
                atomicCAS(p.err, 0u, kErrTimeoutBase | kSiteProdQuant);
                *abort = 1;
                return false;
            }
        }
    }
    fence_acq_rel_gpu();          // the items' writes happen before what follows
    fence_proxy_async_global();   // including the tensor copies of the activation tiles
    return true;
}

// ------------------------------------------------------------- producer --
template <bool kQ6, bool kQuant>
__device__ __forceinline__ void run_producer(const Ctx<kQ6>& cx, const GemmParams& p, const CUtensorMap* tm_x,
                                             const CUtensorMap* tm_e, const CUtensorMap* tm_d) {
    using L = Lay<kQ6>;
    int s = 0, ds = 0;
    uint32_t ph = 0, issued = 0, parity_bits = 0;
    uint32_t dph = 0, d_issued = 0, d_parity_bits = 0;
    bool ok = true;
    int ready_mt = -1;   // token tile whose operand this thread has seen complete
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit w = unit_of<kQ6>(p, u);
        const int mt = w.mt, nt = w.nt;
        if constexpr (kQuant) {   // the operand of tile mt is written by this kernel
            if (mt != ready_mt) {
                if (!quantize_wait(p, mt, cx.abort_flag)) {
                    ok = false;
                    break;
                }
                ready_mt = mt;
            }
            st_release_cta_u32(cx.ready, static_cast<uint32_t>(u) + 1u);   // for the drain's d_a loads
        }
        for (int st = 0; st < w.n_st; ++st) {
            if (!cx.wait(p, L::kBarEmpty + s, ph ^ 1u, kSiteProdEmpty)) {
                ok = false;
                break;
            }
            const int kb_ = st + w.kbase;
            const bool sb_end = kb_ >= 0 && (kb_ + 1) % L::kStPerSb == 0;
            // the last stage of a super-block also brings its d, into the d
            // ring: its slot is taken before any copy of this stage is issued
            if (sb_end && !cx.wait(p, L::kBarDEmpty + ds, dph ^ 1u, kSiteProdD)) {
                ok = false;
                break;
            }
            const uint32_t fb = cx.bar(L::kBarFull + s);
            if (st + w.kbase < 0) {
                if constexpr (!kQ6) {
                    // min-term stage st: depth block st (64 chunks of the
                    // rank-kc product) of E hi and lo into the two A boxes and
                    // of -(dmin*m) hi and lo into the two B boxes, so that the
                    // three products hi*hi, hi*lo and lo*hi come from one load
                    // of each (a box partly past kc reads zeros there)
                    static_assert(L::kStageA >= 2 * L::kBox && L::kStageB >= 2 * L::kBox, "min-term boxes");
                    const int x = 64 * st;
                    mbar_arrive_expect_tx(fb, 4 * L::kBox);
                    tma_load_3d(cx.a(s), tm_e, fb, x, 128 * mt, 0);
                    tma_load_3d(cx.a(s) + L::kBox, tm_e, fb, x, 128 * mt, 1);
                    tma_load_3d(cx.b(s), tm_d, fb, x, 128 * nt, 0);
                    tma_load_3d(cx.b(s) + L::kBox, tm_d, fb, x, 128 * nt, 1);
                }
            } else {
                const int kb = kb_;
                mbar_arrive_expect_tx(fb, L::kStageA + L::kStageNib + L::kStageHi + L::kStageSc);
#pragma unroll
                for (int i = 0; i < L::kCh / 2; ++i)
                    tma_load_2d(cx.a(s) + L::kBox * i, tm_x, fb, 64 * (kb * (L::kCh / 2) + i), 128 * mt);
                const int64_t rec = static_cast<int64_t>(nt) * p.kc + L::kCh * kb;
                bulk_load(cx.base + L::kOffNib + L::kStageNib * s, p.nib + rec * 128 * 16, L::kStageNib, fb);
                if constexpr (kQ6) {   // high quant bits, and two scales per row and chunk
                    bulk_load(cx.base + L::kOffHi + L::kStageHi * s, p.q6hi + rec * 128 * 8, L::kStageHi, fb);
                    bulk_load(cx.base + L::kOffSc + L::kStageSc * s, p.sc + rec * 128 * 2, L::kStageSc, fb);
                } else {
                    bulk_load(cx.base + L::kOffSc + L::kStageSc * s, p.sc + rec * 128, L::kStageSc, fb);
                }
                if (sb_end) {
                    const uint32_t dfb = cx.bar(L::kBarDFull + ds);
                    mbar_arrive_expect_tx(dfb, L::kSlotD);
                    bulk_load(cx.base + L::kOffD + L::kSlotD * ds,
                              p.dsb + (static_cast<int64_t>(nt) * p.ksb + kb / L::kStPerSb) * 128, L::kSlotD, dfb);
                    d_issued |= 1u << ds;
                    d_parity_bits = (d_parity_bits & ~(1u << ds)) | (dph << ds);
                    advance_d<kQ6>(ds, dph);
                }
            }
            issued |= 1u << s;
            parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
            advance<kQ6>(s, ph);
        }
    }
    if (!ok) {   // let every copy this thread started land before the CTA exits
        for (int i = 0; i < L::kStages; ++i)
            if ((issued >> i) & 1u) mbar_wait_quiet(cx.bar(L::kBarFull + i), (parity_bits >> i) & 1u, p.timeout_cycles);
        for (int i = 0; i < L::kDRing; ++i)
            if ((d_issued >> i) & 1u)
                mbar_wait_quiet(cx.bar(L::kBarDFull + i), (d_parity_bits >> i) & 1u, p.timeout_cycles);
    }
}

// ----------------------------------------------------------- MMA issuer --
// TMEM holds four 128-column accumulators in two groups (group g: columns
// 256 g .. 256 g + 255).  One group use is one 16 KB box of a main stage, two
// chunks of 32 k (chunk h of the box accumulates into column 256 g + 128 h),
// or, at the start of a unit with min-term stages, all of its min-term stages
// (Z accumulates into the group's first accumulator).  One commit hands a
// whole group to the drain, and the drain hands it back with one arrival per
// warp.
template <bool kQ6>
__device__ __forceinline__ void run_mma(const Ctx<kQ6>& cx, const GemmParams& p) {
    using L = Lay<kQ6>;
    int s = 0, g = 0;
    uint32_t ph = 0, gph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit w = unit_of<kQ6>(p, u);
        for (int st = 0; st < w.n_st; ++st) {
            const int kb = st + w.kbase;
            // the min-term group is acquired at the unit's first stage, a main
            // stage's groups (one per two chunks) below
            if (st == 0 && kb < 0 && !cx.wait(p, L::kBarAccEmpty + g, gph ^ 1u, kSiteMmaAccEmpty)) {
                ok = false;
                break;
            }
            if (!cx.wait(p, L::kBarFull + s, ph, kSiteMmaFull)) {
                ok = false;
                break;
            }
            // the converters' arrival is awaited on every stage, min-term stages
            // included: a stage is then never refilled before they have passed it
            if (!cx.wait(p, L::kBarConv + s, ph, kSiteMmaConv)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (kb < 0) {
                if constexpr (!kQ6) {   // hi*hi, hi*lo and lo*hi over the block's 64 of depth
                    const uint32_t tg = cx.tmem + 256u * static_cast<uint32_t>(g);
                    const uint64_t ah = sw128_kmajor_desc(cx.a(s)), al = sw128_kmajor_desc(cx.a(s) + L::kBox);
                    const uint64_t bh = sw128_kmajor_desc(cx.b(s)), bl = sw128_kmajor_desc(cx.b(s) + L::kBox);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // K = 64 in four K16 steps of 32 B
                        tc_mma_f16(tg, ah + 2u * kk, bh + 2u * kk, kIdescMin, (st | kk) != 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tg, ah + 2u * kk, bl + 2u * kk, kIdescMin, 1u);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) tc_mma_f16(tg, al + 2u * kk, bh + 2u * kk, kIdescMin, 1u);
                }
                tc_commit(cx.bar(L::kBarEmpty + s));
                if (kb == -1) {   // Z complete: the group goes to the drain
                    tc_commit(cx.bar(L::kBarAccFull + g));
                    if (++g == 2) {
                        g = 0;
                        gph ^= 1u;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < L::kCh / 2; ++j) {   // box j: chunks 2j and 2j+1, one group
                    if (!cx.wait(p, L::kBarAccEmpty + g, gph ^ 1u, kSiteMmaAccEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_kmajor_desc(cx.a(s) + L::kBox * j);
                    const uint64_t bd = sw128_kmajor_desc(cx.b(s) + L::kBox * j);
                    const uint32_t tg = cx.tmem + 256u * static_cast<uint32_t>(g);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t tj = tg + 128u * h;
                        if constexpr (kQ6) {   // fp16: the sh plane, then the sl plane, into one accumulator
                            const uint64_t bl = sw128_kmajor_desc(cx.b(s) + L::kStageB / 2);
                            tc_mma_f16(tj, ad + 4u * h, bd + 4u * h, kIdescMain, 0u);
                            tc_mma_f16(tj, ad + 4u * h + 2u, bd + 4u * h + 2u, kIdescMain, 1u);
                            tc_mma_f16(tj, ad + 4u * h, bl + 4u * h, kIdescMain, 1u);
                            tc_mma_f16(tj, ad + 4u * h + 2u, bl + 4u * h + 2u, kIdescMain, 1u);
                        } else {
                            tc_mma_f16(tj, ad + 4u * h, bd + 4u * h, kIdescMain, 0u);
                            tc_mma_f16(tj, ad + 4u * h + 2u, bd + 4u * h + 2u, kIdescMain, 1u);
                        }
                    }
                    tc_commit(cx.bar(L::kBarAccFull + g));
                    if (++g == 2) {
                        g = 0;
                        gph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(cx.bar(L::kBarEmpty + s));   // the drain reads nothing of the main ring
            }
            advance<kQ6>(s, ph);
        }
    }
    // every MMA this thread issued has finished before the CTA tears down
    tc_commit(cx.bar(L::kBarDrain));
    mbar_wait_quiet(cx.bar(L::kBarDrain), 0u, p.timeout_cycles);
}

// ------------------------------------------------------------ converters --
// Q6_K: row r of stage s.  Each weight's exact integer a = sc * (q - 32) is
// split by its scale: sc = sh + sl with sl = sc & 7 and sh = sc - sl, a
// multiple of 8.  Both parts are exact fp16 integers: sh * (q - 32) is 8 times
// a product of magnitude <= 16 * 32 = 512, and |sl * (q - 32)| <= 224.  The two
// fp16 planes go to the two halves of the B tile, so that two MMAs per 16 k add
// (sh + sl) * (q - 32) * qa = a * qa into the accumulator; with
// |sh * v| + |sl * v| <= 4096 every partial sum of a 32-k chunk stays below
// 32 * 4096 * 127 < 2^24: the chunk integer is exact.  A pair of weights is
// built as fp16(64 + q), the bit pattern 0x5400 | q << 4, straight from the
// packed words, and each plane is one fused multiply-add
// (64 + q) * s - 96 * s = s * (q - 32): exact, since 96 * s and the result are
// fp16 integers.
template <bool kQ6>
__device__ __forceinline__ void convert_q6(const Ctx<kQ6>& cx, int s, int r, uint32_t rx, uint32_t row_off) {
    using L = Lay<kQ6>;
    const uint8_t* lo = cx.sbase + L::kOffNib + L::kStageNib * s;
    const uint8_t* hi = cx.sbase + L::kOffHi + L::kStageHi * s;
    const uint8_t* scs = cx.sbase + L::kOffSc + L::kStageSc * s;
    uint8_t* bh = cx.sbase + L::kOffB + L::kStageB * s + row_off;   // the sh plane
    uint8_t* bl = bh + L::kStageB / 2;                                 // the sl plane
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 wl = *reinterpret_cast<const uint4*>(lo + (h * 128 + r) * 16);
        const uint2 wh = *reinterpret_cast<const uint2*>(hi + (h * 128 + r) * 8);
        const uint32_t scp = *reinterpret_cast<const uint16_t*>(scs + (h * 128 + r) * 2);
        __half2 sh2[2], sl2[2], ch2[2], cl2[2];   // per 16-weight sub-block: the two parts and -96 times them
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int sc = static_cast<int8_t>((scp >> (8 * b)) & 0xFFu);
            const int sl = sc & 7, sh = sc - sl;
            sh2[b] = __half2half2(__int2half_rn(sh));
            sl2[b] = __half2half2(__int2half_rn(sl));
            ch2[b] = __half2half2(__int2half_rn(-96 * sh));
            cl2[b] = __half2half2(__int2half_rn(-96 * sl));
        }
        const uint32_t lw[4] = {wl.x, wl.y, wl.z, wl.w};
        const uint32_t hw[4] = {wh.x, wh.x >> 2, wh.y, wh.y >> 2};
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // 8-k group i of chunk h
            const int b = i >> 1;
            uint32_t oh[4], ol[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                // the pair k = 2jj, 2jj+1: low nibbles at bits 4jj and 16+4jj of the
                // quant word, 2-bit high fields at the same places of the shifted
                // high-bit word; moved to mantissa bits 4-9.  The stored field is
                // u = q ^ 32, so bit 9 is flipped with the exponent bits in one step.
                const uint32_t lf = jj == 0 ? (lw[i] << 4) : (lw[i] >> (4 * jj - 4));
                const uint32_t hf = jj < 2 ? (hw[i] << (8 - 4 * jj)) : (hw[i] >> (4 * jj - 8));
                const uint32_t raw = (lf & 0x00F000F0u) | ((hf & 0x03000300u) ^ 0x56005600u);
                const __half2 v = *reinterpret_cast<const __half2*>(&raw);   // 64 + q
                const __half2 ph = __hfma2(v, sh2[b], ch2[b]);              // sh * (q - 32)
                const __half2 pl = __hfma2(v, sl2[b], cl2[b]);              // sl * (q - 32)
                oh[jj] = *reinterpret_cast<const uint32_t*>(&ph);
                ol[jj] = *reinterpret_cast<const uint32_t*>(&pl);
            }
            const uint32_t g = static_cast<uint32_t>(4 * h + i);
            *reinterpret_cast<uint4*>(bh + ((g ^ rx) << 4)) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
            *reinterpret_cast<uint4*>(bl + ((g ^ rx) << 4)) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
        }
    }
}

// Each thread owns one od row r of the tile.  For chunk h of the stage it
// reads the row's 16 B of quants (4 words, one per 8-k group) and its sc,
// and writes four 16-B granules of fp16 sc*q into row r of the B tile at the
// 128-B-swizzled positions (granule g of row r lands at g ^ (r & 7)).  A
// group of 8 consecutive lanes covers 8 consecutive rows: the 16-B reads are
// contiguous and the granule writes fall in 8 distinct bank quads.
template <bool kQ6>
__device__ __forceinline__ void run_converter(const Ctx<kQ6>& cx, const GemmParams& p, int ci, int lane) {
    using L = Lay<kQ6>;
    const int r = ci * 32 + lane;
    const uint32_t rx = static_cast<uint32_t>(r & 7);
    const uint32_t row_off = static_cast<uint32_t>(r >> 3) * 1024u + rx * 128u;
    const __half2 neg1024 = __float2half2_rn(-1024.0f);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit w = unit_of<kQ6>(p, u);
        for (int st = 0; st < w.n_st; ++st) {
            if (!cx.warp_wait(p, L::kBarFull + s, ph, kSiteConvFull)) {
                ok = false;
                break;
            }
            if (st + w.kbase < 0) {
                // min-term stage: nothing to convert, but arrive anyway so that
                // every stage barrier completes exactly one phase per ring pass
                // and the MMA's phase bit stays valid for it
                __syncwarp();
                if (lane == 0) mbar_arrive(cx.bar(L::kBarConv + s));
            } else if constexpr (kQ6) {
                convert_q6(cx, s, r, rx, row_off);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(cx.bar(L::kBarConv + s));
            } else {
                const uint8_t* nib = cx.sbase + L::kOffNib + L::kStageNib * s;
                const uint8_t* scs = cx.sbase + L::kOffSc + L::kStageSc * s;
#pragma unroll
                for (int h = 0; h < L::kCh; ++h) {   // chunk h: 64-B half (h & 1) of box h / 2
                    uint8_t* brow = cx.sbase + L::kOffB + L::kStageB * s + L::kBox * (h >> 1) + row_off;
                    const uint4 w = *reinterpret_cast<const uint4*>(nib + (h * 128 + r) * 16);
                    const __half2 sc2 = __half2half2(__ushort2half_rn(static_cast<unsigned short>(scs[h * 128 + r])));
                    const __half2 nsc2 = __hmul2(sc2, neg1024);   // -1024*sc, exact
                    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t o[4];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            // (1024 + q) as an fp16 pair, then (1024+q)*sc - 1024*sc = sc*q
                            // in one fused op: exact, as sc*q <= 945 is an fp16 integer
                            const uint32_t pr = ((words[i] >> (4 * jj)) & 0x000F000Fu) | 0x64006400u;
                            const __half2 v = __hfma2(*reinterpret_cast<const __half2*>(&pr), sc2, nsc2);
                            o[jj] = *reinterpret_cast<const uint32_t*>(&v);
                        }
                        const uint32_t g = static_cast<uint32_t>(4 * (h & 1) + i);
                        *reinterpret_cast<uint4*>(brow + ((g ^ rx) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(cx.bar(L::kBarConv + s));
            }
            advance<kQ6>(s, ph);
        }
    }
}

// -------------------------------------------------------------- epilogue --
// The drain keeps the tile's running Y and the super-block's partial sums P
// in registers (64 + 64 per thread: a token row and 64 output columns).
__device__ __forceinline__ void store_row16(const GemmParams& p, int64_t t, int col, const float* v) {
    if (p.out_bf16) {
        __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y) + t * p.ldy + col;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t*>(&pr);
            }
            *reinterpret_cast<uint4*>(y + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        float* y = static_cast<float*>(p.y) + t * p.ldy + col;
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<float4*>(y + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
}

// ---------------------------------------------- SiLU(gate)*up epilogue --
// h = SiLU(g) * u for the down projection, in a fixed fp32 operation order so
// that the q8 codes it yields are reproducible bit for bit: every step is one
// IEEE operation (the _rn intrinsics are never contracted into FMAs).  With
// t = -g:
//   t > 80:   SiLU = RN(g * 0) = -0
//   t < -87:  SiLU = g
//   else:     SiLU = RN(g * R(RN(1 + E(t))))
//   h = RN(SiLU * u)
// E(t) ~ e^t: Cody and Waite's reduction t = n ln2 + r with ln2 split into
// C1 = 355/512 (n*C1 exact) and C2 = RN(ln2 - C1), the degree-7 Taylor
// polynomial of e^r in Horner form, and an exact scaling by 2^n (within
// 1.2 ulp).  R(s) ~ 1/s: a seed read off the bits of s (0x7EF311C2 minus
// them), then three Newton steps y = RN(y * RN(2 - RN(s * y))) (within 2 ulp
// for s in [1, 6e34]).  Everything is branch-free, so that the compiler can
// interleave the 32 elements of a thread.  Constants: the fp32 roundings of
// log2(e), C1, C2 and 1/j!.
__device__ __forceinline__ float silu_mul_fixed(float g, float u) {
    const float t = -g;
    const float tc = fminf(fmaxf(t, -87.0f), 80.0f);
    const float n = rintf(__fmul_rn(tc, 0x1.715476p+0f));
    const float r = __fsub_rn(__fsub_rn(tc, __fmul_rn(n, 0x1.63p-1f)), __fmul_rn(n, -0x1.bd0106p-13f));
    float p = 0x1.a01a02p-13f;                         // 1/7!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.6c16c2p-10f);   // 1/6!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.111112p-7f);    // 1/5!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-5f);    // 1/4!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-3f);    // 1/3!
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    const float e = __fmul_rn(p, __int_as_float((static_cast<int>(n) + 127) << 23));
    const float s = __fadd_rn(1.0f, e);
    float y = __int_as_float(0x7EF311C2 - __float_as_int(s));
#pragma unroll
    for (int i = 0; i < 3; ++i) y = __fmul_rn(y, __fsub_rn(2.0f, __fmul_rn(s, y)));
    float silu = __fmul_rn(g, y);
    silu = t > 80.0f ? __fmul_rn(g, 0.0f) : silu;
    silu = t < -87.0f ? g : silu;
    return __fmul_rn(silu, u);
}

// Tile end of the gate/up pair GEMM: this thread holds, for token t, the 32
// gate outputs (its columns 0-31) and the 32 up outputs of the same features
// (columns 32-63).  It forms h, quantizes it as one 32-element q8
// block (chunk c of the down projection's input; the same rule as
// q8_quantize_rows: d = RN(amax/127), inv = RN(127/amax),
// qa = clamp(rint_even(RN(h*inv)), -127, 127), d_a = RN16(d), a block with
// amax < 2^-120 is zero) and writes the down projection's operand: fp16 qa,
// fp32 d_a and the hi/lo bf16 split of d_a*ssum.
__device__ __forceinline__ void swiglu_store(const GemmParams& p, int64_t t, int c, const float* gate,
                                             const float* up) {
    float h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) h[i] = silu_mul_fixed(gate[i], up[i]);
    float amax = fabsf(h[0]);
#pragma unroll
    for (int i = 1; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
    const Q8Scale sc = q8_scale(amax);
    int ssum = 0;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const int q0 = q8_code(h[i], sc);
        const int q1 = q8_code(h[i + 1], sc);
        ssum += q0 + q1;
        const __half2 pr = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
        w[i >> 1] = *reinterpret_cast<const uint32_t*>(&pr);
    }
    const int64_t kd = static_cast<int64_t>(p.hkc) * 32;
    uint4* dst = reinterpret_cast<uint4*>(p.hq + t * kd + 32 * c);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    const __half da = sc.da;
    p.hda[((t >> 7) * p.hkc + c) * 128 + (t & 127)] = __half2float(da);
    const float e = __fmul_rn(__half2float(da), static_cast<float>(ssum));   // exact: 11 x <= 13 bits
    const __nv_bfloat16 hi = __float2bfloat16_rn(e);
    const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(e, __bfloat162float(hi)));
    p.he[t * p.hkc + c] = hi;
    p.he[(static_cast<int64_t>(p.m) + t) * p.hkc + c] = lo;
}

// A k-part of a split tile: this warp's 32 x 64 slice of the partial Y to the
// workspace, for the fixup kernel.
__device__ __forceinline__ void store_partial(const GemmParams& p, const float* Y, int slot, int slice, int lane) {
    float4* dst = reinterpret_cast<float4*>(p.part + ((static_cast<int64_t>(slot) * 8 + slice) * 32 + lane) * 64);
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[i] = make_float4(Y[4 * i], Y[4 * i + 1], Y[4 * i + 2], Y[4 * i + 3]);
}

// d_a: through the read-only path when another kernel wrote it, through L2
// when this kernel did (the read-only path keeps no promise for data written
// while the kernel runs).
template <bool kQuant>
__device__ __forceinline__ float load_da(const float* a) {
    if constexpr (kQuant) return __ldcg(a);
    return __ldg(a);
}

// The drain's wait for the producer's word that unit `want - 1` has its
// operand complete (every lane polls; the word only grows).
template <bool kQ6>
__device__ __forceinline__ bool ready_wait(const Ctx<kQ6>& cx, const GemmParams& p, uint32_t want) {
    bool ok = true;
    if (ld_acquire_cta_u32(cx.ready) < want) {
        const long long t0 = clock64();
        while (ld_acquire_cta_u32(cx.ready) < want) {
            __nanosleep(64);
            if (*cx.abort_flag) {
                ok = false;
                break;
            }
            if (static_cast<uint64_t>(clock64() - t0) > p.timeout_cycles) {
                atomicCAS(p.err, 0u, kErrTimeoutBase | kSiteEpiReady);
                *cx.abort_flag = 1;
                ok = false;
                break;
            }
        }
    }
    return __all_sync(0xFFFFFFFFu, ok);
}

// Drain warp e (0..7) reads TMEM lanes 32*(warp%4)..+31 (the lane quadrant
// its warp index allows) and columns 64*(e/4)..+63 of each accumulator: each
// thread owns one token row and 64 output columns.  Per main stage it folds
// both chunks, P += d_a * J (packed fp32 FMA), and hands the group back after
// its last TMEM load; per super-block Y += d * P, with d from the d ring
// (it never waits on or releases a stage of the main ring); per unit Y -> HBM.
template <bool kDump, bool kSwiGLU, bool kQ6, bool kQuant>
__device__ __forceinline__ void run_epilogue(const Ctx<kQ6>& cx, const GemmParams& p, int warp, int e, int lane) {
    using L = Lay<kQ6>;
    const int qd = warp & 3, ch = e >> 2;
    const int row = qd * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    int ds = 0, g = 0;
    uint32_t dph = 0, gph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit w = unit_of<kQ6>(p, u);
        const int mt = w.mt, nt = w.nt;
        const int64_t t = static_cast<int64_t>(mt) * 128 + row;
        const int col0 = nt * 128 + 64 * ch;
        float Y[64], P[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            Y[j] = 0.0f;   // a unit without min-term stages starts at zero
            P[j] = 0.0f;
        }
        // d_a straight from global memory (this thread's token, two chunks per
        // accumulator group), loaded kDaAhead groups ahead so that its latency
        // (the L2 under the GEMM's own load) is hidden: dq holds the next groups'
        // values in order, two per group
        constexpr int kDaAhead = 3;
        const int c_end = L::kCh * (w.kbase + w.n_st);
        const float* dap = p.da + static_cast<int64_t>(mt) * p.kc * 128 + row;   // + 128 * chunk
        if constexpr (kQuant) {
            if (!ready_wait(cx, p, static_cast<uint32_t>(u) + 1u)) {
                ok = false;
                break;
            }
        }
        float dq[2 * kDaAhead];
        {
            const int c0 = L::kCh * max(w.kbase, 0);
#pragma unroll
            for (int i = 0; i < 2 * kDaAhead; ++i) dq[i] = c0 + i < c_end ? load_da<kQuant>(dap + 128 * (c0 + i)) : 0.0f;
        }
        for (int st = 0; st < w.n_st; ++st) {
            const int kb = st + w.kbase;
            if (kb == -1) {   // the min-term group is complete: Y starts at Z
                if (!cx.warp_wait(p, L::kBarAccFull + g, gph, kSiteEpiZ)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tz = cx.tmem + lane_off + 256u * static_cast<uint32_t>(g) + 64u * ch;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t Z[16];
                    tmem_ld16(tz + 16u * q, Z);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) Y[16 * q + j] = __uint_as_float(Z[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(cx.bar(L::kBarAccEmpty + g));
                if (++g == 2) {
                    g = 0;
                    gph ^= 1u;
                }
            } else if (kb >= 0) {
#pragma unroll 1
                for (int j = 0; j < L::kCh / 2; ++j) {   // one accumulator group per two chunks
                    const int c = L::kCh * kb + 2 * j;    // its first chunk
                    const float da0 = dq[0], da1 = dq[1];
#pragma unroll
                    for (int i = 0; i + 2 < 2 * kDaAhead; ++i) dq[i] = dq[i + 2];
                    if (c + 2 * kDaAhead < c_end) {
                        dq[2 * kDaAhead - 2] = load_da<kQuant>(dap + 128 * (c + 2 * kDaAhead));
                        dq[2 * kDaAhead - 1] = load_da<kQuant>(dap + 128 * (c + 2 * kDaAhead + 1));
                    }
                    if (!cx.warp_wait(p, L::kBarAccFull + g, gph, kSiteEpiAccFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tg = cx.tmem + lane_off + 256u * static_cast<uint32_t>(g) + 64u * ch;
                    // eight 16-column pieces (chunk pc / 4, columns 16 (pc % 4)): the
                    // next piece's load is in flight while this one is folded
                    uint32_t Ja[16], Jb[16];
                    tmem_ld16(tg, Ja);
                    tmem_wait_ld16(Ja);
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc) {
                        uint32_t (&Jc)[16] = (pc & 1) ? Jb : Ja;
                        uint32_t (&Jn)[16] = (pc & 1) ? Ja : Jb;
                        if (pc + 1 < 8) tmem_ld16(tg + 128u * ((pc + 1) >> 2) + 16u * ((pc + 1) & 3), Jn);
                        const float da = pc < 4 ? da0 : da1;
                        const int q = pc & 3;
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 2)
                            ffma2_ordered(P[16 * q + jj], P[16 * q + jj + 1], da, da, __uint_as_float(Jc[jj]),
                                          __uint_as_float(Jc[jj + 1]));
                        if (kDump && t < p.m) {
#pragma unroll 4
                            for (int jj = 0; jj < 16; ++jj)
                                p.dbg[(t * p.n + col0 + 16 * q + jj) * p.kc + c + (pc >> 2)] = __uint_as_float(Jc[jj]);
                        }
                        if (pc + 1 < 8) tmem_wait_ld16(Jn);
                        if (pc == 6) {   // both accumulators read: the group goes back to the MMA
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(cx.bar(L::kBarAccEmpty + g));
                        }
                    }
                    if (++g == 2) {
                        g = 0;
                        gph ^= 1u;
                    }
                }
                if (!ok) break;
                if ((kb + 1) % L::kStPerSb == 0) {   // super-block done: Y += d * P, d from the d ring
                    if (!cx.warp_wait(p, L::kBarDFull + ds, dph, kSiteEpiD)) {
                        ok = false;
                        break;
                    }
                    const float* dv = reinterpret_cast<const float*>(cx.sbase + L::kOffD + L::kSlotD * ds) + 64 * ch;
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
                        const float4 d4 = *reinterpret_cast<const float4*>(dv + j);
                        Y[j] = fmaf(d4.x, P[j], Y[j]);
                        Y[j + 1] = fmaf(d4.y, P[j + 1], Y[j + 1]);
                        Y[j + 2] = fmaf(d4.z, P[j + 2], Y[j + 2]);
                        Y[j + 3] = fmaf(d4.w, P[j + 3], Y[j + 3]);
                    }
#pragma unroll
                    for (int j = 0; j < 64; ++j) P[j] = 0.0f;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(cx.bar(L::kBarDEmpty + ds));
                    advance_d<kQ6>(ds, dph);
                }
            }
        }
        if (!ok) break;
        if (w.slot >= 0) {   // a k-part of a split tile: its partial Y, finished by the fixup kernel
            store_partial(p, Y, w.slot, qd * 2 + ch, lane);
        } else if constexpr (kSwiGLU) {
            // the 64 columns are 32 gate and 32 up outputs of the down
            // projection's input chunk c = 2 nt + ch
            const int c = 2 * nt + ch;
            if (t < p.m)
                swiglu_store(p, t, c, Y, Y + 32);
            else   // padding token of the last 128-token tile: scale 0
                p.hda[((t >> 7) * p.hkc + c) * 128 + (t & 127)] = 0.0f;
        } else if (t < p.m) {
#pragma unroll
            for (int q = 0; q < 4; ++q) store_row16(p, t, col0 + 16 * q, Y + 16 * q);
        }
    }
}

// kDump: also write every per-chunk accumulator to p.dbg (test hook build).
// kSwiGLU: gate/up pair weights; the tile end writes the down projection's
// q8 operand of SiLU(gate)*up instead of Y.
// kQ6: Q6_K weights (Q6Layout), two fp16 weight planes per stage.
// kQuant: fp32 activations (p.xf), quantized into the workspace by the kernel.
template <bool kDump, bool kSwiGLU, bool kQ6, bool kQuant>
__global__ void __launch_bounds__(kThreads, 1)
    q4k_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_e,
                    const __grid_constant__ CUtensorMap tm_d, const GemmParams p) {
    using L = Lay<kQ6>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    Ctx<kQ6> cx;
    cx.base = base;
    cx.sbase = smem_raw + (base - raw);
    cx.abort_flag = reinterpret_cast<volatile int*>(cx.sbase + L::kOffMisc + 4);
    cx.ready = base + L::kOffMisc + 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(cx.bar(L::kBarFull + s), 1);
            mbar_init(cx.bar(L::kBarConv + s), 4);
            mbar_init(cx.bar(L::kBarEmpty + s), 1);
        }
        for (int i = 0; i < L::kDRing; ++i) {
            mbar_init(cx.bar(L::kBarDFull + i), 1);
            mbar_init(cx.bar(L::kBarDEmpty + i), 8);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(cx.bar(L::kBarAccFull + b), 1);
            mbar_init(cx.bar(L::kBarAccEmpty + b), 8);
        }
        mbar_init(cx.bar(L::kBarDrain), 1);
        *cx.abort_flag = 0;
        *reinterpret_cast<volatile uint32_t*>(cx.sbase + L::kOffMisc + 8) = 0u;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(base + L::kOffMisc, 512);
    if (warp == 1 && lane == 0) {
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_e);
        prefetch_tmap(&tm_d);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cx.tmem = *reinterpret_cast<volatile uint32_t*>(cx.sbase + L::kOffMisc);
    // launched with programmatic dependent launch: the set-up above overlaps
    // the previous kernel's tail; its results (the activation operand) are
    // read, and Y or the workspace written, only after it has completed
    griddep_wait();

    // registers are re-split per warpgroup: the drain holds 128 live values
    // per thread, the producer, MMA and converter roles need far fewer
    if (warp < 4) {
        regs_dec<kRegsCtl>();
        if (warp == 0) {
            if (lane == 0) run_producer<kQ6, kQuant>(cx, p, &tm_x, &tm_e, &tm_d);
            __syncwarp();
        } else if (warp == 1) {
            if (lane == 0) run_mma<kQ6>(cx, p);
            __syncwarp();
        } else if constexpr (kQuant) {   // warps 2 and 3: the items the first wave does not need
            quantize_items<1>(p, p.q_early + (blockIdx.x + gridDim.x - p.q_early % gridDim.x) % gridDim.x,
                              p.q_items, 2, warp - 2, lane, 2u);
        }
    } else if (warp < 8) {
        regs_dec<kRegsConv>();
        run_converter<kQ6>(cx, p, warp - 4, lane);
    } else {
        regs_inc<kRegsDrain>();
        // the first wave's items, before the first accumulator can arrive
        if constexpr (kQuant) quantize_items<4>(p, blockIdx.x, p.q_early, 8, warp - 8, lane, 1u);
        run_epilogue<kDump, kSwiGLU, kQ6, kQuant>(cx, p, warp, warp - 8, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(cx.tmem, 512);
    }
}

// Finishes the k-split tail tiles.  For every element the parts' partial
// values are added in part order (the sum does not depend on which part ran
// where or finished first); then the tile is finished as a whole tile's
// epilogue would finish it.  Work layout: tail tile, slice e (2 x row
// quadrant + column half, as the GEMM stores them), row r of the slice.
__device__ __forceinline__ const float* part_row(const GemmParams& p, int tail, int pp, int e, int r) {
    return p.part + ((static_cast<int64_t>(tail * p.split + pp) * 8 + e) * 32 + r) * 64;
}

// Y: one thread per 4 consecutive columns of a row (16 per row).
__global__ void __launch_bounds__(256) split_fixup_kernel(const GemmParams p) {
    griddep_launch_dependents();   // programmatic dependent launch: the GEMM's partials
    griddep_wait();                // are read only once it has completed
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    const int g = static_cast<int>(gid & 15), r = static_cast<int>((gid >> 4) & 31), e = static_cast<int>((gid >> 9) & 7);
    const int64_t tail = gid >> 12;
    if (tail >= p.num_tiles - p.full_tiles) return;
    const int tile = p.full_tiles + static_cast<int>(tail);
    const int mt = p.nt_fast ? tile / p.n_tiles : tile % p.m_tiles;
    const int nt = p.nt_fast ? tile % p.n_tiles : tile / p.m_tiles;
    const int64_t t = static_cast<int64_t>(mt) * 128 + (e >> 1) * 32 + r;
    if (t >= p.m) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int pp = 0; pp < p.split; ++pp) {
        const float4 v = reinterpret_cast<const float4*>(part_row(p, static_cast<int>(tail), pp, e, r))[g];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    const int64_t col = static_cast<int64_t>(nt) * 128 + 64 * (e & 1) + 4 * g;
    if (p.out_bf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.y) + t * p.ldy + col) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(p.y) + t * p.ldy + col) = acc;
    }
}

// SiLU(gate)*up operand: one warp per row of a slice; lane l adds columns
// 2l and 2l+1 (gate outputs in lanes 0-15, the matching up outputs in lanes
// 16-31), then lanes 0-15 form h and quantize the 32-element block with the
// same operations as the whole-tile epilogue (amax and ssum are exact in any
// order), so the operand bits are those of an unsplit tile with these sums.
__global__ void __launch_bounds__(256) split_fixup_swiglu_kernel(const GemmParams p) {
    griddep_launch_dependents();   // programmatic dependent launch: the GEMM's partials
    griddep_wait();                // are read only once it has completed
    const int64_t wid = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int r = static_cast<int>(wid & 31), e = static_cast<int>((wid >> 5) & 7);
    const int64_t tail = wid >> 8;
    if (tail >= p.num_tiles - p.full_tiles) return;
    const int tile = p.full_tiles + static_cast<int>(tail);
    const int mt = p.nt_fast ? tile / p.n_tiles : tile % p.m_tiles;
    const int nt = p.nt_fast ? tile % p.n_tiles : tile / p.m_tiles;
    const int64_t t = static_cast<int64_t>(mt) * 128 + (e >> 1) * 32 + r;
    const int c = 2 * nt + (e & 1);
    if (t >= p.m) {   // padding token of the last 128-token tile: scale 0
        if (lane == 0) p.hda[((t >> 7) * p.hkc + c) * 128 + (t & 127)] = 0.0f;
        return;
    }
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int pp = 0; pp < p.split; ++pp) {
        const float2 v = reinterpret_cast<const float2*>(part_row(p, static_cast<int>(tail), pp, e, r))[lane];
        acc.x += v.x;
        acc.y += v.y;
    }
    constexpr unsigned kFull = 0xFFFFFFFFu;
    const float u0 = __shfl_down_sync(kFull, acc.x, 16), u1 = __shfl_down_sync(kFull, acc.y, 16);
    const bool gl = lane < 16;
    const float h0 = gl ? silu_mul_fixed(acc.x, u0) : 0.0f;
    const float h1 = gl ? silu_mul_fixed(acc.y, u1) : 0.0f;
    float amax = fmaxf(fabsf(h0), fabsf(h1));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    amax = __shfl_sync(kFull, amax, 0);
    const Q8Scale sc = q8_scale(amax);
    const int q0 = gl ? q8_code(h0, sc) : 0;
    const int q1 = gl ? q8_code(h1, sc) : 0;
    int ssum = q0 + q1;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) ssum += __shfl_xor_sync(kFull, ssum, o);
    if (gl) {
        const __half2 pr = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
        const int64_t kd = static_cast<int64_t>(p.hkc) * 32;
        *reinterpret_cast<__half2*>(p.hq + t * kd + 32 * c + 2 * lane) = pr;
    }
    if (lane == 0) {
        const __half da = sc.da;
        p.hda[((t >> 7) * p.hkc + c) * 128 + (t & 127)] = __half2float(da);
        const float ev = __fmul_rn(__half2float(da), static_cast<float>(ssum));
        const __nv_bfloat16 hi = __float2bfloat16_rn(ev);
        const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(ev, __bfloat162float(hi)));
        p.he[t * p.hkc + c] = hi;
        p.he[(static_cast<int64_t>(p.m) + t) * p.hkc + c] = lo;
    }
}

// Bounded-wait self-test: one CTA waits on a barrier nothing completes.
__global__ void selftest_wait_kernel(unsigned* err, uint64_t timeout_cycles) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(smem_u32(&bar), 0u, &abort_flag, timeout_cycles, err, 0x20u);
    __syncthreads();
}

template <bool kDump, bool kSwiGLU, bool kQ6, bool kQuant>
cudaError_t launch_variant(const CUtensorMap& tm_x, const CUtensorMap& tm_e, const CUtensorMap& tm_d,
                           const GemmParams& p, int grid, cudaStream_t s) {
    static std::atomic<bool> attr_set[64];   // zero at start; a race only repeats the call
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    constexpr size_t smem = Lay<kQ6>::kSmemBytes;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(q4k_gemm_kernel<kDump, kSwiGLU, kQ6, kQuant>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    // in-kernel quantization: CTAs wait for items other CTAs quantize, so all
    // of them must be resident together (a cooperative launch, refused rather
    // than started if they cannot be)
    return launch_pdl_coop(q4k_gemm_kernel<kDump, kSwiGLU, kQ6, kQuant>, kQuant, dim3(grid), dim3(kThreads), smem, s,
                           tm_x, tm_e, tm_d, p);
}

}  // namespace

cudaError_t launch_gemm(const CUtensorMap& tm_x, const CUtensorMap& tm_e, const CUtensorMap& tm_d,
                        const GemmParams& p, int grid, cudaStream_t s) {
    if (p.hq && (p.dbg || p.q6)) return cudaErrorInvalidValue;
    if (p.xf) {   // in-kernel quantization: plain Q4_K weights only
        if (p.dbg || p.q6 || p.hq) return cudaErrorInvalidValue;
        return launch_variant<false, false, false, true>(tm_x, tm_e, tm_d, p, grid, s);
    }
    if (p.q6)
        return p.dbg ? launch_variant<true, false, true, false>(tm_x, tm_e, tm_d, p, grid, s)
                     : launch_variant<false, false, true, false>(tm_x, tm_e, tm_d, p, grid, s);
    if (p.hq) return launch_variant<false, true, false, false>(tm_x, tm_e, tm_d, p, grid, s);
    return p.dbg ? launch_variant<true, false, false, false>(tm_x, tm_e, tm_d, p, grid, s)
                 : launch_variant<false, false, false, false>(tm_x, tm_e, tm_d, p, grid, s);
}

cudaError_t launch_split_fixup(const GemmParams& p, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(p.num_tiles - p.full_tiles) * 8 * 32;   // slice rows
    if (rows <= 0) return cudaSuccess;
    if (p.hq)   // a warp per row
        return launch_pdl(split_fixup_swiglu_kernel, dim3(static_cast<unsigned>((rows * 32 + 255) / 256)), dim3(256), 0,
                          s, p);
    return launch_pdl(split_fixup_kernel, dim3(static_cast<unsigned>((rows * 16 + 255) / 256)), dim3(256), 0, s,
                      p);   // 16 threads per row
}

cudaError_t launch_selftest_wait(unsigned* err, uint64_t timeout_cycles, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(err, timeout_cycles);
    return cudaGetLastError();
}

}  // namespace q4k

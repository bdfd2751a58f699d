// Small-M (decode-sized) Q4_K x q8 product: m <= 16 tokens.
//
// The same arithmetic as the GEMM ("34 · r31 — q-major sda scale-read
// repack", §1-§2: per 32-k chunk an exact integer dot product, then the
// two-term rescale d_a*(d*sc)*sum(q*qa) + d_a*ssum*(-dmin*m)), but with so few
// tokens the product is bound by reading the packed weights from HBM, not by
// the tensor cores.  So it runs on the CUDA cores: the integer dot products
// with dp4a on 4-bit quants unpacked to bytes, the rescale in fp32.
//
// One CTA per 16 od rows (grid = n / 16), 256 threads.  Lane l of warp w owns
// row l % 16 and super-blocks s with s % 16 == 2 * w + l / 16, so a half-warp
// reads 16 consecutive rows' 16-B quant records of one chunk (256 contiguous
// bytes).  For each super-block the half-warp first copies the activations
// it needs (q8 bytes, d_a and ssum of the super-block's 8 chunks, for every
// token) into its own shared-memory stage with 16-B loads, while the quants
// of the next super-block are already on their way into registers; all 16
// lanes then read the stage (broadcast).  The 16 partial sums of a row are
// added in shared memory in a fixed order (deterministic), then stored.  The
// kernel is launched with programmatic dependent launch, so that its quants
// stream into L2 while the kernel before it finishes.
//
// With fp32 activations (kQuant, up to 4 tokens) the stage is filled by
// quantizing them in place of the copy: every CTA quantizes the activations of the super-blocks
// it reads, exactly as the stand-alone q8 quantizer does (same fp32
// operations, so the same q8, d_a and ssum bits), which saves that kernel's
// launch and its round trip through HBM.  The fp32 rows are re-read by every
// CTA from L2 (4 B per element instead of 1), a small cost next to the weights
// at decode sizes.
//
// Per thread and chunk: J[t] = sum_{k in chunk} q[k] * qa[t][k] (exact,
// dp4a), P[t] += d_a[t] * (sc * J[t]) (sc*J < 2^22 is exact in fp32),
// Z[t] += (d_a[t] * ssum[t]) * (-dmin * m) (both factors exact in fp32); per
// super-block Y[t] += d * P[t].
#include <atomic>
#include <cuda_bf16.h>
#include <algorithm>
#include <cuda_fp16.h>

#include "q4k_internal.h"
#include "q4k_gemv.h"
#include "q4k_ptx.cuh"
#include "q8_rule.cuh"
#include "q4k_unpack.cuh"

namespace q4k {
namespace {

constexpr int kRows = 16;      // od rows per CTA
constexpr int kParts = 16;     // super-block shares per row (2 per warp)
constexpr int kThreads = 256;
constexpr size_t kPersistMaxSmem = 220 * 1024;   // persistent form: activations + partial sums

// Activations of one super-block for M tokens.
template <int M>
struct Stage {
    int4 qa[M][16];   // q8 bytes of the 256 k
    uint4 da[M];      // d_a of the 8 chunks (f16 bits)
    uint4 ss[M];      // ssum of the 8 chunks
};

template <int M>
constexpr size_t gemv_smem_bytes() {
    return kParts * sizeof(Stage<M>) > kParts * M * kRows * sizeof(float) ? kParts * sizeof(Stage<M>)
                                                                           : kParts * M * kRows * sizeof(float);
}

// 8 chunks' quants, sc and m of one (row, super-block)
struct SbWeights {
    uint4 q[8];
    uint32_t scm[8];   // sc | m << 8
};

__device__ __forceinline__ void load_weights(const GemvParams& p, int64_t nt, int64_t r, int sb, SbWeights& w) {
    const int64_t rec0 = (nt * p.kc + 8 * sb) * 128 + r;   // chunk 8*sb of this row
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        w.q[j] = __ldg(reinterpret_cast<const uint4*>(p.nib) + rec0 + 128 * j);
        w.scm[j] = static_cast<uint32_t>(__ldg(p.sc + rec0 + 128 * j)) |
                   (static_cast<uint32_t>(__ldg(p.mq + rec0 + 128 * j)) << 8);
    }
}

// Quantize one token's 256 activations of a super-block into the stage.  Lane
// hl of the half-warp takes k = 16 hl .. 16 hl + 15, half of chunk hl / 2; the
// chunk's amax and ssum are completed with the partner lane hl ^ 1.  Rounding
// as in the stand-alone quantizer ("34 · r31 — q-major sda scale-read
// repack", §1 gives the block format; the order is ours): d = RN32(amax/127),
// inv = RN32(127/amax), qa = clamp(rint_even(RN32(x*inv)), -127, 127),
// d_a = RN16(d), and a block with amax < 2^-120 is a zero block.
template <int M>
__device__ __forceinline__ void quantize_to_stage(const float* __restrict__ x, unsigned hmask, int hl, int t,
                                                  Stage<M>& st) {
    const float4* src = reinterpret_cast<const float4*>(x) + 4 * hl;
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 f = __ldg(src + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
    }
    float amax = fabsf(v[0]);
#pragma unroll
    for (int i = 1; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(hmask, amax, 1));
    const Q8Scale sc = q8_scale(amax);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    int s = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int q = q8_code(v[i], sc);
        s += q;
        w[i >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (i & 3));
    }
    s += __shfl_xor_sync(hmask, s, 1);
    st.qa[t][hl] = make_int4(static_cast<int>(w[0]), static_cast<int>(w[1]), static_cast<int>(w[2]),
                             static_cast<int>(w[3]));
    if ((hl & 1) == 0) {
        reinterpret_cast<uint16_t*>(&st.da[t])[hl >> 1] = __half_as_ushort(sc.da);
        reinterpret_cast<int16_t*>(&st.ss[t])[hl >> 1] = static_cast<int16_t>(s);
    }
}

template <int M, bool kQuant>
__global__ void __launch_bounds__(kThreads, kQuant ? 2 : 1) q4k_gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Stage<M>* stages = reinterpret_cast<Stage<M>*>(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hl = lane & 15;                    // row within the CTA / lane within the half-warp
    const int part = 2 * warp + (lane >> 4);     // super-block share
    const int64_t o = static_cast<int64_t>(blockIdx.x) * kRows + hl;
    const int64_t nt = o >> 7, r = o & 127;
    const int kc = p.kc, ksb = p.ksb, m = p.m;
    Stage<M>& st = stages[part];

    // Launched with programmatic dependent launch: while the previous kernel
    // in the stream (normally the activation quantization) still runs, pull
    // this CTA's quants (16 rows x 16 B per chunk, 256 contiguous bytes) from
    // HBM into L2, then wait for that kernel before reading activations.
    griddep_launch_dependents();
    {
        const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRows;
        const int64_t tile0 = row0 >> 7, r0 = row0 & 127;
        for (int c = threadIdx.x; c < kc; c += kThreads)
            prefetch_l2(p.nib + ((tile0 * kc + c) * 128 + r0) * 16, kRows * 16);
    }
    griddep_wait();

    float acc[M];
#pragma unroll
    for (int t = 0; t < M; ++t) acc[t] = 0.0f;

    // Every lane runs the same number of rounds (the two half-warps of a warp
    // may have different numbers of super-blocks): the warp-wide __syncwarp
    // below is then reached by all 32 lanes; a lane without a super-block in
    // a round only takes part in the synchronisation.
    const int rounds = (ksb + kParts - 1) / kParts;
    SbWeights cur, nxt;
    if (part < ksb) load_weights(p, nt, r, part, cur);
    for (int round = 0; round < rounds; ++round) {
        const int sb = part + round * kParts;
        const bool active = sb < ksb;
        if (!active) {   // nothing to do in this pass but the two warp barriers
            __syncwarp();
            __syncwarp();
            continue;
        }
        // stage this super-block's activations (the half-warp shares them)
        if constexpr (kQuant) {
            // the next weights are requested first: the quantization waits on its loads
            if (sb + kParts < ksb) load_weights(p, nt, r, sb + kParts, nxt);
            const unsigned hmask = 0xFFFFu << (lane & 16);
#pragma unroll 2
            for (int t = 0; t < M; ++t)
                if (t < m) quantize_to_stage<M>(p.xf + t * p.ldx + 256 * sb, hmask, hl, t, st);
        } else {
#pragma unroll
            for (int t = 0; t < M; ++t)
                if (t < m) st.qa[t][hl] = __ldg(reinterpret_cast<const int4*>(p.q8 + t * p.ldq + 256 * sb) + hl);
            if (hl < m && hl < M) {
                st.da[hl] = __ldg(reinterpret_cast<const uint4*>(p.da + hl * kc + 8 * sb));
                st.ss[hl] = __ldg(reinterpret_cast<const uint4*>(p.ssum + hl * kc + 8 * sb));
            }
            if (sb + kParts < ksb) load_weights(p, nt, r, sb + kParts, nxt);   // in flight during this one
        }
        const int64_t srec = (nt * ksb + sb) * 128 + r;
        const float d = __ldg(p.dsb + srec);
        const float dmin = __ldg(p.dmn + srec);
        __syncwarp();
        float P[M], Z[M];
#pragma unroll
        for (int t = 0; t < M; ++t) {
            P[t] = 0.0f;
            Z[t] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t q[8];
            unpack_group(cur.q[j].x, q[0], q[1]);
            unpack_group(cur.q[j].y, q[2], q[3]);
            unpack_group(cur.q[j].z, q[4], q[5]);
            unpack_group(cur.q[j].w, q[6], q[7]);
            const int sc = static_cast<int>(cur.scm[j] & 0xFFu);
            const float nm = -(dmin * static_cast<float>(cur.scm[j] >> 8));   // exact: f16 value x 6-bit m
#pragma unroll
            for (int t = 0; t < M; ++t) {
                if (t < m) {
                    const int4 a0 = st.qa[t][2 * j], a1 = st.qa[t][2 * j + 1];
                    int J = __dp4a(static_cast<int>(q[0]), a0.x, 0);
                    J = __dp4a(static_cast<int>(q[1]), a0.y, J);
                    J = __dp4a(static_cast<int>(q[2]), a0.z, J);
                    J = __dp4a(static_cast<int>(q[3]), a0.w, J);
                    J = __dp4a(static_cast<int>(q[4]), a1.x, J);
                    J = __dp4a(static_cast<int>(q[5]), a1.y, J);
                    J = __dp4a(static_cast<int>(q[6]), a1.z, J);
                    J = __dp4a(static_cast<int>(q[7]), a1.w, J);
                    const float da =
                        __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(&st.da[t])[j]));
                    const float ss = static_cast<float>(reinterpret_cast<const int16_t*>(&st.ss[t])[j]);
                    P[t] = fmaf(da, static_cast<float>(sc * J), P[t]);
                    Z[t] = fmaf(da * ss, nm, Z[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < M; ++t) acc[t] = fmaf(d, P[t], acc[t]) + Z[t];
        __syncwarp();   // the stage is read by every lane before the next super-block overwrites it
        cur = nxt;
    }

    // add the 16 shares of each row in a fixed order (the stages are free now)
    __syncthreads();
    float* red = reinterpret_cast<float*>(smem_raw);   // [kParts][M][kRows]
#pragma unroll
    for (int t = 0; t < M; ++t) red[(part * M + t) * kRows + hl] = acc[t];
    __syncthreads();
    for (int i = threadIdx.x; i < M * kRows; i += kThreads) {
        const int t = i / kRows, rr = i % kRows;
        if (t >= m) continue;
        float v = 0.0f;
#pragma unroll
        for (int s = 0; s < kParts; ++s) v += red[(s * M + t) * kRows + rr];
        const int64_t oo = static_cast<int64_t>(blockIdx.x) * kRows + rr;
        if (p.out_bf16)
            static_cast<__nv_bfloat16*>(p.y)[t * p.ldy + oo] = __float2bfloat16_rn(v);
        else
            static_cast<float*>(p.y)[t * p.ldy + oo] = v;
    }
}

// ------------------------------------------------------- persistent form --
// The same arithmetic with the activations staged once per CTA: the grid is
// one or two CTAs per SM, each CTA first copies (q8 input) or quantizes (fp32
// input) all m x k activations into shared memory, then walks 16-row groups
// g = blockIdx.x, blockIdx.x + gridDim.x, ...  A thread's weights for the
// next (row group, super-block) are in flight while it computes the current
// one, across row-group boundaries too, so the weight stream does not stop
// between groups.  Per group the 16 shares of a row are added in shared
// memory in a fixed order, as above.
struct PersistSmem {
    size_t act, da, ss, red, total;   // byte offsets: q8 [m][k], d_a f16 [m][kc], ssum [m][kc], partial sums
    __host__ __device__ static size_t a16(size_t v) { return (v + 15) / 16 * 16; }
    __host__ __device__ PersistSmem(int mslots, int k) {
        const size_t kc = static_cast<size_t>(k) / 32;
        act = 0;
        da = a16(static_cast<size_t>(mslots) * k);
        ss = da + a16(static_cast<size_t>(mslots) * kc * 2);
        red = ss + a16(static_cast<size_t>(mslots) * kc * 2);
        total = red + static_cast<size_t>(kParts) * mslots * kRows * 4;
    }
};

// One 32-element q8 block quantized by one thread (the rule of the activation
// quantizer: d = RN(amax/127), inv = RN(127/amax), qa = clamp(rint_even(
// RN(x*inv)), -127, 127), d_a = RN16(d), zero block below 2^-120).
__device__ __forceinline__ void quantize_block_to(const float* __restrict__ src, int8_t* dst, uint16_t* da,
                                                  int16_t* ss) {
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
    uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    int s = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int q = q8_code(v[i], sc);
        s += q;
        w[i >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (i & 3));
    }
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    *da = __half_as_ushort(sc.da);
    *ss = static_cast<int16_t>(s);
}

// Stage all m x k activations of the call in shared memory: copy the q8 SoA
// (16-byte pieces), or quantize fp32 rows one 32-element block per thread.
template <bool kQuant>
__device__ __forceinline__ void stage_activations(const GemvParams& p, int8_t* act, uint16_t* sda, int16_t* sss) {
    const int kc = p.kc, m = p.m, k = p.k;
    if constexpr (kQuant) {
        for (int i = threadIdx.x; i < m * kc; i += kThreads) {
            const int t = i / kc, c = i - t * kc;
            quantize_block_to(p.xf + static_cast<int64_t>(t) * p.ldx + 32 * c, act + static_cast<int64_t>(t) * k + 32 * c,
                              sda + t * kc + c, sss + t * kc + c);
        }
    } else {
        const int v16 = k / 16, s8 = kc / 8;   // 16-B pieces of a q8 row and of a scale row
        for (int i = threadIdx.x; i < m * v16; i += kThreads) {
            const int t = i / v16, j = i - t * v16;
            reinterpret_cast<int4*>(act + static_cast<int64_t>(t) * k)[j] =
                __ldg(reinterpret_cast<const int4*>(p.q8 + t * p.ldq) + j);
        }
        for (int i = threadIdx.x; i < m * s8; i += kThreads) {
            const int t = i / s8, j = i - t * s8;
            reinterpret_cast<uint4*>(sda + t * kc)[j] = __ldg(reinterpret_cast<const uint4*>(p.da + t * kc) + j);
            reinterpret_cast<uint4*>(sss + t * kc)[j] = __ldg(reinterpret_cast<const uint4*>(p.ssum + t * kc) + j);
        }
    }
}

// Add the 16 shares of each row of group g in a fixed order and store them.
template <int M>
__device__ __forceinline__ void reduce_store(const GemvParams& p, float* red, const float (&acc)[M], int part, int hl,
                                             int g) {
    __syncthreads();   // the previous group's sums have been read
#pragma unroll
    for (int t = 0; t < M; ++t) red[(part * M + t) * kRows + hl] = acc[t];
    __syncthreads();
    for (int i = threadIdx.x; i < M * kRows; i += kThreads) {
        const int t = i / kRows, rr = i % kRows;
        if (t >= p.m) continue;
        float v = 0.0f;
#pragma unroll
        for (int s2 = 0; s2 < kParts; ++s2) v += red[(s2 * M + t) * kRows + rr];
        const int64_t oo = static_cast<int64_t>(g) * kRows + rr;
        if (p.out_bf16)
            static_cast<__nv_bfloat16*>(p.y)[t * p.ldy + oo] = __float2bfloat16_rn(v);
        else
            static_cast<float*>(p.y)[t * p.ldy + oo] = v;
    }
}

template <int M, bool kQuant>
__global__ void __launch_bounds__(kThreads, M == 1 ? 2 : 1) q4k_gemv_persistent_kernel(const GemvParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hl = lane & 15;
    const int part = 2 * warp + (lane >> 4);
    const int kc = p.kc, ksb = p.ksb, m = p.m, k = p.k;
    const int groups = p.n / kRows;
    const PersistSmem L(M, k);
    int8_t* act = reinterpret_cast<int8_t*>(smem_raw + L.act);
    uint16_t* sda = reinterpret_cast<uint16_t*>(smem_raw + L.da);
    int16_t* sss = reinterpret_cast<int16_t*>(smem_raw + L.ss);
    float* red = reinterpret_cast<float*>(smem_raw + L.red);

    // programmatic dependent launch: this CTA's first row group streams into
    // L2 while the previous kernel finishes
    griddep_launch_dependents();
    if (blockIdx.x < groups) {
        const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRows;
        const int64_t tile0 = row0 >> 7, r0 = row0 & 127;
        for (int c = threadIdx.x; c < kc; c += kThreads)
            prefetch_l2(p.nib + ((tile0 * kc + c) * 128 + r0) * 16, kRows * 16);
    }
    griddep_wait();

    // the first weights are requested before the activations are staged
    const int rounds = (ksb + kParts - 1) / kParts;
    SbWeights cur, nxt;
    int g = blockIdx.x;
    if (g < groups && part < ksb) {
        const int64_t o = static_cast<int64_t>(g) * kRows + hl;
        load_weights(p, o >> 7, o & 127, part, cur);
    }
    stage_activations<kQuant>(p, act, sda, sss);
    __syncthreads();

    for (; g < groups; g += gridDim.x) {
        const int64_t o = static_cast<int64_t>(g) * kRows + hl;
        const int64_t nt = o >> 7, r = o & 127;
        const int gn = g + gridDim.x;   // this CTA's next row group
        float acc[M];
#pragma unroll
        for (int t = 0; t < M; ++t) acc[t] = 0.0f;
        for (int round = 0; round < rounds; ++round) {
            const int sb = part + round * kParts;
            if (sb >= ksb) continue;   // no barrier inside the round: nothing to keep in step
            if (sb + kParts < ksb) {
                load_weights(p, nt, r, sb + kParts, nxt);
            } else if (gn < groups) {
                const int64_t on = static_cast<int64_t>(gn) * kRows + hl;
                load_weights(p, on >> 7, on & 127, part, nxt);
            }
            const int64_t srec = (nt * ksb + sb) * 128 + r;
            const float d = __ldg(p.dsb + srec);
            const float dmin = __ldg(p.dmn + srec);
            float P[M], Z[M];
#pragma unroll
            for (int t = 0; t < M; ++t) {
                P[t] = 0.0f;
                Z[t] = 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t q[8];
                unpack_group(cur.q[j].x, q[0], q[1]);
                unpack_group(cur.q[j].y, q[2], q[3]);
                unpack_group(cur.q[j].z, q[4], q[5]);
                unpack_group(cur.q[j].w, q[6], q[7]);
                const int sc = static_cast<int>(cur.scm[j] & 0xFFu);
                const float nm = -(dmin * static_cast<float>(cur.scm[j] >> 8));   // exact: f16 value x 6-bit m
                const int c = 8 * sb + j;
#pragma unroll
                for (int t = 0; t < M; ++t) {
                    if (t < m) {
                        const int4* a = reinterpret_cast<const int4*>(act + static_cast<int64_t>(t) * k + 32 * c);
                        const int4 a0 = a[0], a1 = a[1];
                        int J = __dp4a(static_cast<int>(q[0]), a0.x, 0);
                        J = __dp4a(static_cast<int>(q[1]), a0.y, J);
                        J = __dp4a(static_cast<int>(q[2]), a0.z, J);
                        J = __dp4a(static_cast<int>(q[3]), a0.w, J);
                        J = __dp4a(static_cast<int>(q[4]), a1.x, J);
                        J = __dp4a(static_cast<int>(q[5]), a1.y, J);
                        J = __dp4a(static_cast<int>(q[6]), a1.z, J);
                        J = __dp4a(static_cast<int>(q[7]), a1.w, J);
                        const float da = __half2float(__ushort_as_half(sda[t * kc + c]));
                        const float ss = static_cast<float>(sss[t * kc + c]);
                        P[t] = fmaf(da, static_cast<float>(sc * J), P[t]);
                        Z[t] = fmaf(da * ss, nm, Z[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < M; ++t) acc[t] = fmaf(d, P[t], acc[t]) + Z[t];
            cur = nxt;
        }
        reduce_store<M>(p, red, acc, part, hl, g);
    }
}

// --------------------------------------------------------------- Q6_K --
// Q6_K weights (w = d*sc*(q-32), one signed 8-bit sc per 16 weights) in the
// persistent form.  Per 32-k chunk the exact integer
//   I = sc_0 * sum_{k<16} (q-32)*qa + sc_1 * sum_{k>=16} (q-32)*qa
// (|I| <= 32*128*32*127 < 2^24, exact in fp32), then P += d_a*I per chunk
// and Y += d*P per super-block.  The packed 6-bit u = q ^ 32 is q - 32 in
// 6-bit two's complement: low nibbles and the 2 high bits are put back into
// bytes and sign-extended, and dp4a multiplies signed bytes.
struct SbWeightsQ6 {
    uint4 lo[8];
    uint2 hi[8];
    uint32_t sc[8];   // the chunk's two i8 scales (bytes 0 and 1)
};

__device__ __forceinline__ void load_weights_q6(const GemvParams& p, int64_t nt, int64_t r, int sb, SbWeightsQ6& w) {
    const int64_t rec0 = (nt * p.kc + 8 * sb) * 128 + r;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        w.lo[j] = __ldg(reinterpret_cast<const uint4*>(p.nib) + rec0 + 128 * j);
        w.hi[j] = __ldg(reinterpret_cast<const uint2*>(p.q6hi) + rec0 + 128 * j);
        w.sc[j] = __ldg(reinterpret_cast<const uint16_t*>(p.sc) + rec0 + 128 * j);
    }
}

template <int M, bool kQuant>
__global__ void __launch_bounds__(kThreads, M == 1 ? 2 : 1) q6k_gemv_persistent_kernel(const GemvParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hl = lane & 15;
    const int part = 2 * warp + (lane >> 4);
    const int kc = p.kc, ksb = p.ksb, m = p.m, k = p.k;
    const int groups = p.n / kRows;
    const PersistSmem L(M, k);
    int8_t* act = reinterpret_cast<int8_t*>(smem_raw + L.act);
    uint16_t* sda = reinterpret_cast<uint16_t*>(smem_raw + L.da);
    int16_t* sss = reinterpret_cast<int16_t*>(smem_raw + L.ss);
    float* red = reinterpret_cast<float*>(smem_raw + L.red);

    griddep_launch_dependents();
    if (blockIdx.x < groups) {
        const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRows;
        const int64_t tile0 = row0 >> 7, r0 = row0 & 127;
        for (int c = threadIdx.x; c < kc; c += kThreads) {
            prefetch_l2(p.nib + ((tile0 * kc + c) * 128 + r0) * 16, kRows * 16);
            prefetch_l2(p.q6hi + ((tile0 * kc + c) * 128 + r0) * 8, kRows * 8);
        }
    }
    griddep_wait();

    const int rounds = (ksb + kParts - 1) / kParts;
    SbWeightsQ6 cur, nxt;
    int g = blockIdx.x;
    if (g < groups && part < ksb) {
        const int64_t o = static_cast<int64_t>(g) * kRows + hl;
        load_weights_q6(p, o >> 7, o & 127, part, cur);
    }
    stage_activations<kQuant>(p, act, sda, sss);
    __syncthreads();

    for (; g < groups; g += gridDim.x) {
        const int64_t o = static_cast<int64_t>(g) * kRows + hl;
        const int64_t nt = o >> 7, r = o & 127;
        const int gn = g + gridDim.x;
        float acc[M];
#pragma unroll
        for (int t = 0; t < M; ++t) acc[t] = 0.0f;
        for (int round = 0; round < rounds; ++round) {
            const int sb = part + round * kParts;
            if (sb >= ksb) continue;
            if (sb + kParts < ksb) {
                load_weights_q6(p, nt, r, sb + kParts, nxt);
            } else if (gn < groups) {
                const int64_t on = static_cast<int64_t>(gn) * kRows + hl;
                load_weights_q6(p, on >> 7, on & 127, part, nxt);
            }
            const float d = __ldg(p.dsb + (nt * ksb + sb) * 128 + r);
            float P[M];
#pragma unroll
            for (int t = 0; t < M; ++t) P[t] = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t v[8];
                unpack_q6(cur.lo[j].x, cur.hi[j].x, v[0], v[1]);
                unpack_q6(cur.lo[j].y, cur.hi[j].x >> 2, v[2], v[3]);
                unpack_q6(cur.lo[j].z, cur.hi[j].y, v[4], v[5]);
                unpack_q6(cur.lo[j].w, cur.hi[j].y >> 2, v[6], v[7]);
                const int sc0 = static_cast<int>(static_cast<int8_t>(cur.sc[j] & 0xFFu));
                const int sc1 = static_cast<int>(static_cast<int8_t>((cur.sc[j] >> 8) & 0xFFu));
                const int c = 8 * sb + j;
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
                        const float da = __half2float(__ushort_as_half(sda[t * kc + c]));
                        P[t] = fmaf(da, static_cast<float>(sc0 * J0 + sc1 * J1), P[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < M; ++t) acc[t] = fmaf(d, P[t], acc[t]);
            cur = nxt;
        }
        reduce_store<M>(p, red, acc, part, hl, g);
    }
}

template <int M, bool kQuant>
cudaError_t launch_q6k_gemv_m(const GemvParams& p, cudaStream_t s) {
    static std::atomic<bool> attr_set[64];   // zero at start; a race only repeats the call
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = PersistSmem(M, p.k).total;
    if (smem > kPersistMaxSmem) return cudaErrorInvalidValue;   // the caller checks the size first
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(q6k_gemv_persistent_kernel<M, kQuant>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kPersistMaxSmem));
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q6k_gemv_persistent_kernel<M, kQuant>, kThreads,
                                                          smem)) != cudaSuccess)
        return e;
    const int groups = static_cast<int>(p.n / kRows);
    const int grid = std::max(1, std::min(groups, std::max(1, per_sm) * sms));
    return launch_pdl(q6k_gemv_persistent_kernel<M, kQuant>, dim3(grid), dim3(kThreads), smem, s, p);
}

// Launch the persistent form when its activations fit in shared memory and
// there are enough row groups; otherwise leave *launched false.
template <int M, bool kQuant>
cudaError_t launch_gemv_persistent(const GemvParams& p, cudaStream_t s, bool* launched) {
    *launched = false;
    static std::atomic<size_t> smem_set[64];   // zero at start; a race only repeats the call
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = PersistSmem(M, p.k).total;
    if (smem > kPersistMaxSmem) return cudaSuccess;   // too large: the caller uses the other form
    if (smem_set[dev].load(std::memory_order_acquire) < smem) {   // raise the limit once per size class
        e = cudaFuncSetAttribute(q4k_gemv_persistent_kernel<M, kQuant>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kPersistMaxSmem));
        if (e != cudaSuccess) return e;
        smem_set[dev].store(kPersistMaxSmem, std::memory_order_release);
    }
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q4k_gemv_persistent_kernel<M, kQuant>, kThreads,
                                                          smem)) != cudaSuccess)
        return e;
    const int groups = static_cast<int>(p.n / kRows);
    const int slots = std::max(1, per_sm) * sms;
    // Staging all activations pays off only when a CTA then works through
    // several row groups (measured: with one group per CTA the per-group form
    // is faster); quantizing them costs more than copying, so it needs more.
    if (groups <= (kQuant ? 2 : 1) * slots) return cudaSuccess;
    const int grid = std::min(groups, slots);
    *launched = true;
    return launch_pdl(q4k_gemv_persistent_kernel<M, kQuant>, dim3(grid), dim3(kThreads), smem, s, p);
}

template <int M, bool kQuant>
cudaError_t launch_gemv_m(const GemvParams& p, cudaStream_t s) {
    static std::atomic<bool> attr_set[64];   // zero at start; a race only repeats the call
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    constexpr size_t smem = gemv_smem_bytes<M>();
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(q4k_gemv_kernel<M, kQuant>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.n / kRows));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, q4k_gemv_kernel<M, kQuant>, p);
}

template <int M, bool kQuant>
cudaError_t launch_gemv_any(const GemvParams& p, cudaStream_t s) {
    bool launched = false;
    const cudaError_t e = launch_gemv_persistent<M, kQuant>(p, s, &launched);
    if (e != cudaSuccess || launched) return e;
    return launch_gemv_m<M, kQuant>(p, s);
}

cudaError_t launch_gemv_q8(const GemvParams& p, cudaStream_t s) {
    if (p.m <= 1) return launch_gemv_any<1, false>(p, s);
    if (p.m <= 2) return launch_gemv_any<2, false>(p, s);
    if (p.m <= 4) return launch_gemv_any<4, false>(p, s);
    if (p.m <= 8) return launch_gemv_any<8, false>(p, s);
    return launch_gemv_any<16, false>(p, s);
}

}  // namespace

bool gemv_q6k_fits(int m, int64_t k) {
    const int slots = m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : m <= 8 ? 8 : 16;   // the kernel's token slots
    return PersistSmem(slots, static_cast<int>(k)).total <= kPersistMaxSmem;
}

cudaError_t launch_gemv_q6k(const GemvParams& p, cudaStream_t s) {
    bool launched = false;
    const cudaError_t e = launch_gemv_stream(p, s, &launched);
    if (e != cudaSuccess || launched) return e;
    if (p.xf) {   // in-kernel quantization: up to 4 tokens (the caller's limit)
        if (p.m <= 1) return launch_q6k_gemv_m<1, true>(p, s);
        if (p.m <= 2) return launch_q6k_gemv_m<2, true>(p, s);
        if (p.m <= 4) return launch_q6k_gemv_m<4, true>(p, s);
        return cudaErrorInvalidValue;
    }
    if (p.m <= 1) return launch_q6k_gemv_m<1, false>(p, s);
    if (p.m <= 2) return launch_q6k_gemv_m<2, false>(p, s);
    if (p.m <= 4) return launch_q6k_gemv_m<4, false>(p, s);
    if (p.m <= 8) return launch_q6k_gemv_m<8, false>(p, s);
    return launch_q6k_gemv_m<16, false>(p, s);
}

cudaError_t launch_gemv(const GemvParams& p, cudaStream_t s) {
    bool launched = false;
    const cudaError_t e = launch_gemv_stream(p, s, &launched);
    if (e != cudaSuccess || launched) return e;
    if (!p.xf) return launch_gemv_q8(p, s);
    // in-kernel quantization is built for up to 4 tokens (the caller's limit)
    if (p.m <= 1) return launch_gemv_any<1, true>(p, s);
    if (p.m <= 2) return launch_gemv_any<2, true>(p, s);
    if (p.m <= 4) return launch_gemv_any<4, true>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace q4k

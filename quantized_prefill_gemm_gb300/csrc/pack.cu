// Load-time repack of canonical Q4_K blocks into the GEMM's tiled layout.
//
// Q4_K semantics: 256-weight super-blocks with f16 d and dmin, eight 32-weight
// sub-blocks with 6-bit sc and 6-bit m, 4-bit q; w = d*sc*q - dmin*m
// ("34 · r31 — q-major sda scale-read repack", §2: the B side of the rescale
// is the per-(chunk, od row) pair d*sc and -dmin*m).  Byte layout read as the
// public GGUF Q4_K arrangement: d, dmin (f16), 12 bytes holding the sixteen
// 6-bit scale/min fields, 128 bytes of quants (pair of sub-blocks 2p, 2p+1 in
// the low / high nibbles of bytes 32p..32p+31).
//
// Output (q4k_layout.h): per (128-row tile, chunk) records of 16 B of quants
// in the order the GEMM's converter expands them, the sc bytes, the fp32 d of
// each super-block, -(dmin*m) split into two bf16 planes for the min-term
// GEMM, and for the small-M path the m bytes and the fp32 dmin of each
// super-block.  One thread per (od row, super-block); runs once per weight
// matrix.
//
// Gate/up pairs (for the SiLU(gate)*up epilogue): the packed matrix has 2n
// rows; packed row R of tile T = R / 128 takes, for j = (R % 128) / 32 and
// i = R % 32, row 64 T + 32 (j / 2) + i of the gate (j even) or up (j odd)
// matrix.  So each half of a 128-row tile holds 32 gate rows and the 32 up
// rows of the same outputs, side by side.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4k_internal.h"
#include "q4k_layout.h"

namespace q4k {
namespace {

constexpr int kThreadsPerBlock = 128;

// blocks: [n][k/256] canonical blocks; up: null, or the up matrix of a gate
// (blocks) / up pair, n then being the packed row count 2 x (rows of each).
__global__ void __launch_bounds__(kThreadsPerBlock) pack_kernel(const uint8_t* __restrict__ blocks,
                                                                const uint8_t* __restrict__ up, int64_t n,
                                                                int64_t k, uint8_t* __restrict__ packed,
                                                                int64_t off_sc, int64_t off_dsb, int64_t off_ndm,
                                                                int64_t off_mq, int64_t off_dmn) {
    const int64_t ksb = k / 256, kc = k / 32;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= n * ksb) return;
    const int64_t o = idx / ksb, sb = idx % ksb;
    const uint8_t* blk = blocks + idx * 144;
    if (up) {
        const int64_t j = (o & 127) >> 5;
        const int64_t src = 64 * (o >> 7) + 32 * (j >> 1) + (o & 31);
        blk = ((j & 1) ? up : blocks) + (src * ksb + sb) * 144;
    }

    const uint32_t head = *reinterpret_cast<const uint32_t*>(blk);
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(head & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(head >> 16)));

    uint8_t s[12];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(blk + 4 + 4 * i);
#pragma unroll
        for (int b = 0; b < 4; ++b) s[4 * i + b] = static_cast<uint8_t>(w >> (8 * b));
    }
    int scv[8], mv[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        scv[j] = s[j] & 63;
        mv[j] = s[j + 4] & 63;
        scv[j + 4] = (s[j + 8] & 15) | ((s[j] >> 6) << 4);
        mv[j + 4] = (s[j + 8] >> 4) | ((s[j + 4] >> 6) << 4);
    }

    const int64_t nt = o >> 7, r = o & 127;
    uint8_t* nib = packed;
    uint8_t* scp = packed + off_sc;
    float* dsb = reinterpret_cast<float*>(packed + off_dsb);
    __nv_bfloat16* ndm = reinterpret_cast<__nv_bfloat16*>(packed + off_ndm);
    uint8_t* mqp = packed + off_mq;
    float* dmn = reinterpret_cast<float*>(packed + off_dmn);

    for (int j = 0; j < 8; ++j) {   // sub-block = chunk c of this super-block
        const int64_t c = sb * 8 + j;
        const uint8_t* qs = blk + 16 + 32 * (j >> 1);
        const int shift = (j & 1) ? 4 : 0;
        uint32_t words[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // k-group of 8 inside the chunk
            uint32_t w = 0;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const uint32_t q_even = (qs[8 * i + 2 * jj] >> shift) & 15u;
                const uint32_t q_odd = (qs[8 * i + 2 * jj + 1] >> shift) & 15u;
                w |= q_even << (4 * jj);
                w |= q_odd << (16 + 4 * jj);
            }
            words[i] = w;
        }
        const int64_t rec = (nt * kc + c) * 128 + r;
        *reinterpret_cast<uint4*>(nib + rec * 16) = make_uint4(words[0], words[1], words[2], words[3]);
        scp[rec] = static_cast<uint8_t>(scv[j]);
        mqp[rec] = static_cast<uint8_t>(mv[j]);
        const float v = -(dmin * static_cast<float>(mv[j]));   // exact: 11-bit x 6-bit
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
        ndm[o * kc + c] = hi;
        ndm[(n + o) * kc + c] = lo;
    }
    dsb[(nt * ksb + sb) * 128 + r] = d;
    dmn[(nt * ksb + sb) * 128 + r] = dmin;
}

// Q6_K (q6k_blocks layout of the public GGUF format: ql[128], qh[64],
// sc[16] int8, d f16; w = d*sc*(q-32)) -> Q6Layout.  One thread per (row,
// super-block).
__global__ void __launch_bounds__(kThreadsPerBlock) pack_q6k_kernel(const uint8_t* __restrict__ blocks, int64_t n,
                                                                    int64_t k, uint8_t* __restrict__ packed,
                                                                    int64_t off_hi, int64_t off_sc, int64_t off_dsb) {
    const int64_t ksb = k / 256, kc = k / 32;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= n * ksb) return;
    const int64_t o = idx / ksb, sb = idx % ksb;
    const uint8_t* blk = blocks + idx * 210;
    const int64_t nt = o >> 7, r = o & 127;
    for (int j = 0; j < 8; ++j) {   // chunk c = 8 sb + j: weights 32j .. 32j+31 of the super-block
        uint8_t u[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int wi = 32 * j + i;                 // weight index in the super-block
            const int h = wi >> 7, l = wi & 31, part = (wi >> 5) & 3;
            const uint8_t lob = blk[64 * h + l + ((part & 1) ? 32 : 0)];
            const uint8_t hib = blk[128 + 32 * h + l];
            const int q = (((part & 2) ? (lob >> 4) : (lob & 15)) | (((hib >> (2 * part)) & 3) << 4));
            u[i] = static_cast<uint8_t>(q ^ 32);
        }
        uint32_t lw[4], hw[2] = {0u, 0u};
#pragma unroll
        for (int g = 0; g < 4; ++g) {   // 8-k group g: k = 8g .. 8g+7 of the chunk
            uint32_t w = 0;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const uint32_t ue = u[8 * g + 2 * jj], uo = u[8 * g + 2 * jj + 1];
                w |= (ue & 15u) << (4 * jj);
                w |= (uo & 15u) << (16 + 4 * jj);
                hw[g >> 1] |= ((ue >> 4) & 3u) << (4 * jj + 2 * (g & 1));
                hw[g >> 1] |= ((uo >> 4) & 3u) << (16 + 4 * jj + 2 * (g & 1));
            }
            lw[g] = w;
        }
        const int64_t rec = (nt * kc + sb * 8 + j) * 128 + r;
        *reinterpret_cast<uint4*>(packed + rec * 16) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        *reinterpret_cast<uint2*>(packed + off_hi + rec * 8) = make_uint2(hw[0], hw[1]);
        packed[off_sc + rec * 2] = blk[192 + 2 * j];
        packed[off_sc + rec * 2 + 1] = blk[192 + 2 * j + 1];
    }
    const float d = __half2float(__ushort_as_half(
        static_cast<unsigned short>(blk[208] | (static_cast<unsigned>(blk[209]) << 8))));
    reinterpret_cast<float*>(packed + off_dsb)[(nt * ksb + sb) * 128 + r] = d;
}

}  // namespace

cudaError_t launch_pack_q6k(const uint8_t* blocks, int64_t n, int64_t k, uint8_t* packed, cudaStream_t s) {
    const Q6Layout L(n, k);
    const int64_t threads = n * (k / 256);
    if (threads == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((threads + kThreadsPerBlock - 1) / kThreadsPerBlock);
    pack_q6k_kernel<<<grid, kThreadsPerBlock, 0, s>>>(blocks, n, k, packed, L.hi, L.sc, L.dsb);
    return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* blocks, int64_t n, int64_t k, uint8_t* packed, cudaStream_t s) {
    const PackedLayout L(n, k);
    const int64_t threads = n * (k / 256);
    if (threads == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((threads + kThreadsPerBlock - 1) / kThreadsPerBlock);
    pack_kernel<<<grid, kThreadsPerBlock, 0, s>>>(blocks, nullptr, n, k, packed, L.sc, L.dsb, L.ndm, L.mq, L.dmn);
    return cudaGetLastError();
}

cudaError_t launch_pack_pair(const uint8_t* gate, const uint8_t* up, int64_t n, int64_t k, uint8_t* packed,
                             cudaStream_t s) {
    const PackedLayout L(2 * n, k);
    const int64_t threads = 2 * n * (k / 256);
    if (threads == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((threads + kThreadsPerBlock - 1) / kThreadsPerBlock);
    pack_kernel<<<grid, kThreadsPerBlock, 0, s>>>(gate, up, 2 * n, k, packed, L.sc, L.dsb, L.ndm, L.mq, L.dmn);
    return cudaGetLastError();
}

}  // namespace q4k

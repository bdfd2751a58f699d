// Launch wrappers shared by the library's translation units (not exported).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace q4k {

// Launch with programmatic dependent launch: the kernel may start while the
// previous kernel in the stream finishes; it must execute griddepcontrol.wait
// before it touches memory that kernel reads or writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The same, and with `coop` also as a cooperative launch: every CTA of the
// grid is resident at once, or the launch fails.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_coop(void (*kernel)(KArgs...), bool coop, dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = coop ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// 32-k chunks per main stage of the tensor-core GEMM: 4 (128 k) for Q4_K,
// 2 (64 k) for Q6_K, whose stages carry two fp16 weight planes.
__host__ __device__ constexpr int gemm_chunks_per_stage(bool q6) { return q6 ? 2 : 4; }

struct GemmParams {
    const uint8_t* nib;     // packed quants  [nt][kc][128][16 B]
    const uint8_t* sc;      // packed scales  [nt][kc][128]
    const float* dsb;       // super-block d  [nt][ksb][128]
    const float* da;        // token scales   [mp/128][kc][128]
    void* y;                // output [m][ldy]
    float* dbg;             // optional per-chunk accumulators [m][n][kc] (test hook)
    unsigned* err;          // device error word
    uint64_t timeout_cycles;   // bound of every internal wait, in SM clock cycles
    int64_t ldy;
    int m, n, k;
    int kc, ksb;
    int m_tiles, n_tiles, num_tiles;
    int n_zst, n_main;      // min-term stages and main stages per tile
    // Work units: tiles [0, full_tiles) whole, then each remaining tile in
    // `split` parts along k of part_sb super-blocks (part 0 also runs the
    // min-term stages); split == 1 means every tile is whole.
    int full_tiles, split, part_sb, num_units;
    float* part;            // [kMaxSplitUnits][8][32][64] partial tiles (ActLayout)
    int out_bf16;
    // SiLU(gate)*up epilogue (gate/up pair weights, y unused): the down
    // projection's activation operand for kd = n / 2 inputs, in the
    // q4k_act_quantize layout (q4k_layout.h, ActLayout(m, kd))
    __half* hq;             // [m][kd] fp16 qa
    float* hda;             // [mp/128][kd/32][128] d_a
    __nv_bfloat16* he;      // [2][m][kd/32] d_a*ssum hi / lo
    int hkc;                // kd / 32
    // Q6_K weights (Q6Layout: nib = low nibbles, sc = i8 scale pairs,
    // dsb = d) with the fp16 activation operand; no min term
    const uint8_t* q6hi;    // the high quant bits [nt][kc][128][8 B]
    int q6;
    // Tile order: 0 = token tile fastest (tile = nt * m_tiles + mt), 1 = output
    // tile fastest (tile = mt * n_tiles + nt), the order the in-kernel
    // quantization needs (the first wave then reads the first token tiles only).
    int nt_fast;
    // In-kernel quantization (xf set): the kernel writes the activation operand
    // (xq, da, e of the workspace) from fp32 x itself.  Item i = (token tile
    // i / qs, slice i % qs of its kc blocks); item i is quantized by CTA
    // i % gridDim.x, items below q_early at the start by the drain warps, the
    // others alongside the GEMM by the two spare warps.  qflag[mt] counts the
    // finished items of token tile mt under this call's tag qtag.
    const float* xf;        // [m][ldx] fp32, or null (operand already in the workspace)
    int64_t ldx;
    uint16_t* xq_w;         // the workspace's xq, da and e, written by the kernel
    float* da_w;
    __nv_bfloat16* e_w;
    unsigned long long* qflag;   // [m_tiles]
    unsigned long long qtag;     // bits 16-63; the count lives in bits 0-15
    int qs, q_early, q_items;
};

cudaError_t launch_q8_quantize_rows(const float* x, int64_t m, int64_t k, int64_t ldx, int8_t* q8,
                                    uint16_t* da, int16_t* ssum, cudaStream_t s);
// The GEMM operand form in ws (ActLayout): fp16 codes, d_a, and the bf16 hi/lo of d_a * ssum.
cudaError_t launch_act_quantize(const float* x, int64_t m, int64_t k, int64_t ldx, void* ws, cudaStream_t s);
cudaError_t launch_act_from_q8(const int8_t* q8, const uint16_t* da, const int16_t* ssum, int64_t m, int64_t k,
                               int64_t ldq, void* ws, cudaStream_t s);
cudaError_t launch_pack(const uint8_t* blocks, int64_t n, int64_t k, uint8_t* packed, cudaStream_t s);
// Q6_K blocks [n][k/256] x 210 B -> Q6Layout (small-M path)
cudaError_t launch_pack_q6k(const uint8_t* blocks, int64_t n, int64_t k, uint8_t* packed, cudaStream_t s);
// gate and up [n][k/256] blocks each -> one packed matrix of 2n interleaved rows
cudaError_t launch_pack_pair(const uint8_t* gate, const uint8_t* up, int64_t n, int64_t k, uint8_t* packed,
                             cudaStream_t s);
cudaError_t launch_gemm(const CUtensorMap& tm_x, const CUtensorMap& tm_e, const CUtensorMap& tm_d,
                        const GemmParams& p, int grid, cudaStream_t s);
// After a GEMM with split > 1: add each split tile's parts and finish it.
cudaError_t launch_split_fixup(const GemmParams& p, cudaStream_t s);
cudaError_t launch_selftest_wait(unsigned* err, uint64_t timeout_cycles, cudaStream_t s);
// blocks x 256 threads, each warp iters x 8 mma.sync m16n8k32 s8 (peak.cu)
cudaError_t launch_peak_s8(int64_t blocks, int64_t iters, int* sink, cudaStream_t s);

}  // namespace q4k

// Host side of the C ABI declared in include/q4k.h: argument validation,
// buffer layouts, TMA descriptor encoding and kernel launches.  Nothing here
// allocates device memory; only the diagnostics synchronise.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/q4k.h"
#include "q4k_internal.h"
#include "q4k_gemv.h"
#include "q4k_layout.h"

namespace q4k {

// Device-side error word (one per device context).  Host code must not use
// this name as an address: the device address comes from
// cudaGetSymbolAddress, looked up per device with that device current.
__device__ unsigned int g_device_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 4ull * 1000 * 1000 * 1000;   // 4 s per wait
// waits are bounded in SM cycles; 2 cycles per ns keeps the bound >= the
// nominal time at any clock up to 2 GHz (longer at lower clocks)
constexpr uint64_t kCyclesPerNs = 2;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    unsigned* err_word = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

q4k_status from_cuda(cudaError_t e) { return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA; }

// Per-device set-up (first call on each device, with that device current):
// architecture check, SM count, device address of the error word.
q4k_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4K_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return Q4K_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return Q4K_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.sm_count = sms;
        void* p = nullptr;
        if (d.supported) {
            if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return Q4K_ERR_CUDA;
        }
        d.err_word = static_cast<unsigned*>(p);
        d.ready = true;
    }
    if (!d.supported) return Q4K_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return Q4K_OK;
}

q4k_status encoder(EncodeTiledFn* fn) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f)
            return Q4K_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(f);
    }
    *fn = g_encode;
    return Q4K_OK;
}

// Row-major [rows][inner] (times `planes`) tensor, tiles of 64 inner x 128
// rows, 128-byte swizzle, zero fill outside the tensor.
q4k_status encode_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int64_t inner, int64_t rows,
                      int64_t planes) {
    EncodeTiledFn fn = nullptr;
    q4k_status st = encoder(&fn);
    if (st != Q4K_OK) return st;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner * 2), static_cast<cuuint64_t>(inner * rows * 2)};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint32_t rank = planes > 1 ? 3 : 2;
    const CUresult r = fn(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? Q4K_OK : Q4K_ERR_CUDA;
}

// The tag of one GEMM call that quantizes its activations in the kernel: a
// fixed mark in bits 48-63 and a per-process call counter in bits 16-47 (bits
// 0-15 carry the kernel's counts).  The counter starts at a clock-derived
// value, so that a count another process left in reused memory is unlikely to
// carry the same tag either.
unsigned long long next_quant_tag() {
    static std::atomic<uint32_t> counter{
        static_cast<uint32_t>(static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) *
                              2654435761ull)};
    const uint32_t e = counter.fetch_add(1u, std::memory_order_relaxed);
    return (0x51A4ull << 48) | (static_cast<unsigned long long>(e) << 16);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kMaxDim = int64_t(1) << 31;

q4k_status check_act_f32(const float* x, int64_t m, int64_t k, int64_t ldx) {
    if (m < 0 || k <= 0 || m >= kMaxDim || k >= kMaxDim) return Q4K_ERR_SHAPE;
    if (k % 32) return Q4K_ERR_SHAPE;
    if (ldx < k) return Q4K_ERR_SHAPE;
    if (m > 0 && !x) return Q4K_ERR_INVALID_ARG;
    if (m > 0 && (!aligned(x, 16) || ldx % 4)) return Q4K_ERR_ALIGNMENT;
    return Q4K_OK;
}

q4k_status check_gemm_shape(int64_t n, int64_t k, int64_t m) {
    if (n <= 0 || k <= 0 || m < 0 || n >= kMaxDim || k >= kMaxDim || m >= kMaxDim) return Q4K_ERR_SHAPE;
    if (n % kTileN || k % 256) return Q4K_ERR_SHAPE;
    return Q4K_OK;
}

q4k_status check_output(const void* y, int64_t m, int64_t n, int out, int64_t ldy) {
    if (out != Q4K_OUT_F32 && out != Q4K_OUT_BF16) return Q4K_ERR_INVALID_ARG;
    if (ldy < n) return Q4K_ERR_SHAPE;
    if (m > 0 && !y) return Q4K_ERR_INVALID_ARG;
    if (m > 0 && (!aligned(y, 16) || ldy % (out == Q4K_OUT_F32 ? 4 : 8))) return Q4K_ERR_ALIGNMENT;
    return Q4K_OK;
}

// h_ws (gate/up pair weights only): instead of Y, write the down projection's
// operand of SiLU(gate)*up, ActLayout(m, n / 2), there; y, out and ldy are then
// unused.  The caller has checked h_ws.  q6: Q6_K weights (Q6Layout); the
// activation operand in ws has the same fp16 form as for Q4_K.  xf: fp32
// activations [m][ldx] (checked by the caller) that the GEMM kernel quantizes
// into ws itself; without it ws already holds the operand.
q4k_status run_gemm(const void* packed_w, int64_t n, int64_t k, void* ws, size_t ws_bytes, int64_t m, void* y,
                    int out, int64_t ldy, float* dbg, void* h_ws, cudaStream_t stream, bool q6 = false,
                    const float* xf = nullptr, int64_t ldx = 0) {
    q4k_status st = check_gemm_shape(n, k, m);
    if (st != Q4K_OK) return st;
    if (!h_ws && (st = check_output(y, m, n, out, ldy)) != Q4K_OK) return st;
    if (!packed_w || (m > 0 && !ws)) return Q4K_ERR_INVALID_ARG;
    if (!aligned(packed_w, 256) || (m > 0 && !aligned(ws, 256))) return Q4K_ERR_ALIGNMENT;
    const ActLayout A(m, k);
    if (m > 0 && ws_bytes < static_cast<size_t>(A.total)) return Q4K_ERR_WORKSPACE;
    if (m == 0) return Q4K_OK;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != Q4K_OK) return st;

    const PackedLayout W(n, k);
    const Q6Layout W6(n, k);
    const uint8_t* wb = static_cast<const uint8_t*>(packed_w);
    uint8_t* ab = static_cast<uint8_t*>(ws);
    const int64_t kc = k / 32;
    CUtensorMap tm_x, tm_e, tm_d;
    if ((st = encode_map(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ab + A.xq, k,
                         m, 1)) != Q4K_OK)
        return st;
    if (q6) {   // no min term: the min-term maps are not used
        tm_e = tm_x;
        tm_d = tm_x;
    } else {
        if ((st = encode_map(&tm_e, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ab + A.e, kc, m, 2)) != Q4K_OK) return st;
        if ((st = encode_map(&tm_d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, wb + W.ndm, kc, n, 2)) != Q4K_OK) return st;
    }

    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    if (q6) {
        p.nib = wb + W6.lo;
        p.q6hi = wb + W6.hi;
        p.sc = wb + W6.sc;
        p.dsb = reinterpret_cast<const float*>(wb + W6.dsb);
        p.q6 = 1;
    } else {
        p.nib = wb + W.nib;
        p.sc = wb + W.sc;
        p.dsb = reinterpret_cast<const float*>(wb + W.dsb);
    }
    p.da = reinterpret_cast<const float*>(ab + A.da);
    p.y = y;
    p.dbg = dbg;
    p.err = dev->err_word;
    p.timeout_cycles = kDefaultTimeoutNs * kCyclesPerNs;
    p.ldy = ldy;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.kc = static_cast<int>(kc);
    p.ksb = static_cast<int>(k / 256);
    p.m_tiles = static_cast<int>((m + kTileM - 1) / kTileM);
    p.n_tiles = static_cast<int>(n / kTileN);
    p.num_tiles = p.m_tiles * p.n_tiles;
    // min-term stages: one per 64 of depth (hi and lo of both operands)
    p.n_zst = q6 ? 0 : static_cast<int>((kc + 63) / 64);
    p.n_main = static_cast<int>(k / (32 * gemm_chunks_per_stage(q6)));
    p.out_bf16 = out == Q4K_OUT_BF16 ? 1 : 0;
    // Tail balance: after the last full wave of tiles over the SMs, the R
    // remaining tiles are split along k into parts (whole super-blocks) so
    // that R x parts work units occupy the otherwise idle SMs.  The epilogue
    // writes each part's partial tile to the workspace; a small kernel then
    // adds a tile's parts in part order (deterministic) and finishes the tile
    // as usual, so Y, or the SiLU(gate)*up operand, comes from the same fp32
    // sums whichever output the call asks for.  Tiles of fewer than four
    // super-blocks are not split: the fixup launch costs more than the
    // shorter units save (measured: 256 x 512 at 64 tokens, 18.0 -> 15.8 us).
    // A part holds at least two super-blocks: one-super-block parts (the 8
    // leftover tiles of 11008 x 4096 at 2048 tokens in 16 parts) measured
    // slower than 8 parts of two, by their per-unit start and the fixup's
    // reads (the 7B stack 38,983 -> 39,133 tok/s with two).
    p.split = 1;
    p.part_sb = p.ksb;
    p.full_tiles = p.num_tiles;
    const int sms = std::min<int>(dev->sm_count, static_cast<int>(kMaxSplitUnits));
    const int rem = p.num_tiles % sms;
    if (rem > 0) {
        const int parts = std::min(sms / rem, std::max(2, p.ksb / 2));
        if (parts >= 2 && p.ksb >= 4) {
            p.part_sb = (p.ksb + parts - 1) / parts;
            p.split = (p.ksb + p.part_sb - 1) / p.part_sb;
            p.full_tiles = p.num_tiles - rem;
        }
    }
    p.num_units = p.full_tiles + (p.num_tiles - p.full_tiles) * p.split;
    p.part = reinterpret_cast<float*>(ab + A.part);
    if (h_ws) {
        const ActLayout H(m, n / 2);
        uint8_t* hb = static_cast<uint8_t*>(h_ws);
        p.hq = reinterpret_cast<__half*>(hb + H.xq);
        p.hda = reinterpret_cast<float*>(hb + H.da);
        p.he = reinterpret_cast<__nv_bfloat16*>(hb + H.e);
        p.hkc = static_cast<int>(n / 64);
    }
    const int grid = std::min(p.num_units, dev->sm_count);
    if (xf) {   // in-kernel quantization (gemm.cu): items of the operand, counted per token tile
        p.nt_fast = 1;   // output tiles fastest: the first wave reads the first token tiles only
        p.xf = xf;
        p.ldx = ldx;
        p.xq_w = reinterpret_cast<uint16_t*>(ab + A.xq);
        p.da_w = reinterpret_cast<float*>(ab + A.da);
        p.e_w = reinterpret_cast<__nv_bfloat16*>(ab + A.e);
        p.qflag = reinterpret_cast<unsigned long long*>(ab + A.flag);
        p.qtag = next_quant_tag();
        // the last token tile the first wave of units reads; its tiles and the
        // ones before it are cut into about one item per CTA
        const int last = std::min(grid, p.num_units) - 1;
        const int tile = last < p.full_tiles ? last : p.full_tiles + (last - p.full_tiles) / p.split;
        const int mt1 = tile / p.n_tiles;
        p.qs = std::max(1, std::min(p.kc, grid / (mt1 + 1)));
        p.q_items = p.m_tiles * p.qs;
        p.q_early = std::min(p.q_items, (mt1 + 1) * p.qs);
    }
    if ((st = from_cuda(launch_gemm(tm_x, tm_e, tm_d, p, grid, stream))) != Q4K_OK) return st;
    return p.split > 1 ? from_cuda(launch_split_fixup(p, stream)) : Q4K_OK;
}

// Small-M path on the CUDA cores: the packed weights times either the q8 SoA
// (q8 rows, d_a and ssum 16-byte aligned, ldq % 16 == 0) or, when xf is set,
// fp32 activations (16-byte aligned, ldx % 4 == 0) quantized in the kernel.
q4k_status run_gemv(const void* packed_w, int64_t n, int64_t k, const int8_t* q8, const uint16_t* da,
                    const int16_t* ssum, const float* xf, int64_t m, int64_t ldq, void* y, int out, int64_t ldy,
                    cudaStream_t stream) {
    DeviceInfo* dev = nullptr;
    q4k_status st = device_info(&dev);
    if (st != Q4K_OK) return st;
    const PackedLayout W(n, k);
    const uint8_t* wb = static_cast<const uint8_t*>(packed_w);
    GemvParams g;
    std::memset(&g, 0, sizeof(g));
    g.nib = wb + W.nib;
    g.sc = wb + W.sc;
    g.mq = wb + W.mq;
    g.dsb = reinterpret_cast<const float*>(wb + W.dsb);
    g.dmn = reinterpret_cast<const float*>(wb + W.dmn);
    g.q8 = q8;
    g.da = da;
    g.ssum = ssum;
    g.xf = xf;
    g.y = y;
    g.ldq = xf ? 0 : ldq;
    g.ldx = xf ? ldq : 0;
    g.ldy = ldy;
    g.m = static_cast<int>(m);
    g.n = static_cast<int>(n);
    g.k = static_cast<int>(k);
    g.kc = static_cast<int>(k / 32);
    g.ksb = static_cast<int>(k / 256);
    g.out_bf16 = out == Q4K_OUT_BF16 ? 1 : 0;
    return from_cuda(launch_gemv(g, stream));
}

// Where the small-M path keeps the q8 SoA inside a q4k_gemm workspace (token
// counts above kFusedQuantMaxM).
struct SmallMLayout {
    int64_t q8, da, ssum, total;
    SmallMLayout(int64_t m, int64_t k) {
        const int64_t kc = k / 32;
        q8 = 0;
        da = align_up(m * k, 256);
        ssum = align_up(da + m * kc * 2, 256);
        total = align_up(ssum + m * kc * 2, 256);
    }
};

// Up to this many tokens the small-M kernel quantizes fp32 activations itself.
// Every CTA quantizes the whole activation block it reads, so the repeated
// work grows with m; beyond 4 tokens a separate q8 pass is faster.
constexpr int64_t kFusedQuantMaxM = Q4K_FUSED_QUANT_M;

}  // namespace
}  // namespace q4k

using namespace q4k;

extern "C" {

const char* q4k_status_string(int status) {
    switch (status) {
        case Q4K_OK: return "ok";
        case Q4K_ERR_INVALID_ARG: return "invalid argument";
        case Q4K_ERR_SHAPE: return "unsupported shape";
        case Q4K_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
        case Q4K_ERR_WORKSPACE: return "workspace or packed buffer too small";
        case Q4K_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103 (GB300)";
        case Q4K_ERR_CUDA: return "CUDA call failed";
        case Q4K_ERR_TIMEOUT: return "bounded device-side wait timed out";
        default: return "unknown status";
    }
}

int q4k_abi_version(void) { return Q4K_ABI_VERSION; }

q4k_status q8_quantize_rows(const float* x, int64_t m, int64_t k, int64_t ldx, int8_t* q8, uint16_t* da_f16,
                            int16_t* ssum, cudaStream_t stream) {
    q4k_status st = check_act_f32(x, m, k, ldx);
    if (st != Q4K_OK) return st;
    if (m == 0) return Q4K_OK;
    if (!q8 || !da_f16 || !ssum) return Q4K_ERR_INVALID_ARG;
    if (!aligned(q8, 4) || !aligned(da_f16, 2) || !aligned(ssum, 2)) return Q4K_ERR_ALIGNMENT;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != Q4K_OK) return st;
    return from_cuda(launch_q8_quantize_rows(x, m, k, ldx, q8, da_f16, ssum, stream));
}

size_t q4k_packed_bytes(int64_t n, int64_t k) {
    if (n <= 0 || k <= 0 || n % kTileN || k % 256 || n >= kMaxDim || k >= kMaxDim) return 0;
    return static_cast<size_t>(PackedLayout(n, k).total);
}

q4k_status q4k_pack_weights(const void* blocks, int64_t n, int64_t k, void* packed, size_t packed_bytes,
                            cudaStream_t stream) {
    if (n <= 0 || k <= 0 || n % kTileN || k % 256 || n >= kMaxDim || k >= kMaxDim) return Q4K_ERR_SHAPE;
    if (!blocks || !packed) return Q4K_ERR_INVALID_ARG;
    if (!aligned(blocks, 16) || !aligned(packed, 256)) return Q4K_ERR_ALIGNMENT;
    if (packed_bytes < q4k_packed_bytes(n, k)) return Q4K_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    q4k_status st = device_info(&dev);
    if (st != Q4K_OK) return st;
    return from_cuda(launch_pack(static_cast<const uint8_t*>(blocks), n, k, static_cast<uint8_t*>(packed), stream));
}

size_t q4k_swiglu_packed_bytes(int64_t n, int64_t k) {
    if (n <= 0 || n % 64 || n >= kMaxDim / 2) return 0;
    return q4k_packed_bytes(2 * n, k);
}

q4k_status q4k_pack_swiglu_weights(const void* gate_blocks, const void* up_blocks, int64_t n, int64_t k,
                                   void* packed, size_t packed_bytes, cudaStream_t stream) {
    if (n <= 0 || k <= 0 || n % 64 || k % 256 || n >= kMaxDim / 2 || k >= kMaxDim) return Q4K_ERR_SHAPE;
    if (!gate_blocks || !up_blocks || !packed) return Q4K_ERR_INVALID_ARG;
    if (!aligned(gate_blocks, 16) || !aligned(up_blocks, 16) || !aligned(packed, 256)) return Q4K_ERR_ALIGNMENT;
    if (packed_bytes < q4k_swiglu_packed_bytes(n, k)) return Q4K_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    q4k_status st = device_info(&dev);
    if (st != Q4K_OK) return st;
    return from_cuda(launch_pack_pair(static_cast<const uint8_t*>(gate_blocks), static_cast<const uint8_t*>(up_blocks),
                                      n, k, static_cast<uint8_t*>(packed), stream));
}

size_t q4k_act_workspace_bytes(int64_t m, int64_t k) {
    if (m < 0 || k <= 0 || k % 256 || m >= kMaxDim || k >= kMaxDim) return 0;
    return static_cast<size_t>(ActLayout(m, k).total);
}

size_t q4k_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int act) {
    (void)n;
    if (act != Q4K_ACT_F32 && act != Q4K_ACT_Q8) return 0;
    return q4k_act_workspace_bytes(m, k);
}

q4k_status q4k_act_quantize(const float* x, int64_t m, int64_t k, int64_t ldx, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
    q4k_status st = check_act_f32(x, m, k, ldx);
    if (st != Q4K_OK) return st;
    if (k % 256) return Q4K_ERR_SHAPE;
    if (m == 0) return Q4K_OK;
    if (!workspace) return Q4K_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return Q4K_ERR_ALIGNMENT;
    if (workspace_bytes < q4k_act_workspace_bytes(m, k)) return Q4K_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != Q4K_OK) return st;
    return from_cuda(launch_act_quantize(x, m, k, ldx, workspace, stream));
}

q4k_status q4k_act_from_q8(const int8_t* q8, const uint16_t* da_f16, const int16_t* ssum, int64_t m, int64_t k,
                           int64_t ldq, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (m < 0 || k <= 0 || k % 256 || m >= kMaxDim || k >= kMaxDim || ldq < k) return Q4K_ERR_SHAPE;
    if (m == 0) return Q4K_OK;
    if (!q8 || !da_f16 || !ssum || !workspace) return Q4K_ERR_INVALID_ARG;
    if (!aligned(q8, 4) || ldq % 4 || !aligned(da_f16, 2) || !aligned(ssum, 2) || !aligned(workspace, 256))
        return Q4K_ERR_ALIGNMENT;
    if (workspace_bytes < q4k_act_workspace_bytes(m, k)) return Q4K_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    q4k_status st = device_info(&dev);
    if (st != Q4K_OK) return st;
    return from_cuda(launch_act_from_q8(q8, da_f16, ssum, m, k, ldq, workspace, stream));
}

q4k_status q4k_gemm_quantized(const void* packed_w, int64_t n, int64_t k, void* workspace,
                              size_t workspace_bytes, int64_t m, void* y, int out_dtype, int64_t ldy,
                              cudaStream_t stream) {
    return run_gemm(packed_w, n, k, workspace, workspace_bytes, m, y, out_dtype, ldy, nullptr, nullptr, stream);
}

q4k_status q4k_gemm(const void* packed_w, int64_t n, int64_t k, int act, const void* x_or_q8, const void* da_f16,
                    const void* ssum, int64_t m, int64_t ldx, void* y, int out_dtype, int64_t ldy,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    q4k_status st = check_gemm_shape(n, k, m);
    if (st != Q4K_OK) return st;
    if ((st = check_output(y, m, n, out_dtype, ldy)) != Q4K_OK) return st;
    if (!packed_w) return Q4K_ERR_INVALID_ARG;
    if (act != Q4K_ACT_F32 && act != Q4K_ACT_Q8) return Q4K_ERR_INVALID_ARG;
    if (!aligned(packed_w, 256)) return Q4K_ERR_ALIGNMENT;
    if (m >= 1 && m <= Q4K_SMALL_M) {   // decode-sized: CUDA-core path, bound by the weight stream
        if (act == Q4K_ACT_F32) {
            const float* xf = static_cast<const float*>(x_or_q8);
            if ((st = check_act_f32(xf, m, k, ldx)) != Q4K_OK) return st;
            if (m <= kFusedQuantMaxM)   // one launch: the kernel quantizes the activations itself
                return run_gemv(packed_w, n, k, nullptr, nullptr, nullptr, xf, m, ldx, y, out_dtype, ldy, stream);
            const SmallMLayout L(m, k);
            if (!workspace) return Q4K_ERR_INVALID_ARG;
            if (!aligned(workspace, 256)) return Q4K_ERR_ALIGNMENT;
            if (workspace_bytes < static_cast<size_t>(L.total)) return Q4K_ERR_WORKSPACE;
            uint8_t* wsb = static_cast<uint8_t*>(workspace);
            int8_t* q8 = reinterpret_cast<int8_t*>(wsb + L.q8);
            uint16_t* da = reinterpret_cast<uint16_t*>(wsb + L.da);
            int16_t* ss = reinterpret_cast<int16_t*>(wsb + L.ssum);
            st = q8_quantize_rows(xf, m, k, ldx, q8, da, ss, stream);
            if (st != Q4K_OK) return st;
            return run_gemv(packed_w, n, k, q8, da, ss, nullptr, m, k, y, out_dtype, ldy, stream);
        }
        const int8_t* q8 = static_cast<const int8_t*>(x_or_q8);
        if (!q8 || !da_f16 || !ssum) return Q4K_ERR_INVALID_ARG;
        if (ldx < k) return Q4K_ERR_SHAPE;
        if (aligned(q8, 16) && ldx % 16 == 0 && aligned(da_f16, 16) && aligned(ssum, 16))
            return run_gemv(packed_w, n, k, q8, static_cast<const uint16_t*>(da_f16),
                            static_cast<const int16_t*>(ssum), nullptr, m, ldx, y, out_dtype, ldy, stream);
        // other alignments go through the general path below
    }
    if (act == Q4K_ACT_F32) {
        st = q4k_act_quantize(static_cast<const float*>(x_or_q8), m, k, ldx, workspace, workspace_bytes, stream);
    } else {
        st = q4k_act_from_q8(static_cast<const int8_t*>(x_or_q8), static_cast<const uint16_t*>(da_f16),
                             static_cast<const int16_t*>(ssum), m, k, ldx, workspace, workspace_bytes, stream);
    }
    if (st != Q4K_OK) return st;
    return run_gemm(packed_w, n, k, workspace, workspace_bytes, m, y, out_dtype, ldy, nullptr, nullptr, stream);
}

q4k_status q4k_gemm_inkernel_quant(const void* packed_w, int64_t n, int64_t k, const float* x, int64_t m,
                                   int64_t ldx, void* y, int out_dtype, int64_t ldy, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
    q4k_status st = check_gemm_shape(n, k, m);
    if (st != Q4K_OK) return st;
    if ((st = check_output(y, m, n, out_dtype, ldy)) != Q4K_OK) return st;
    if ((st = check_act_f32(x, m, k, ldx)) != Q4K_OK) return st;
    if (!packed_w) return Q4K_ERR_INVALID_ARG;
    if (!aligned(packed_w, 256)) return Q4K_ERR_ALIGNMENT;
    return run_gemm(packed_w, n, k, workspace, workspace_bytes, m, y, out_dtype, ldy, nullptr, nullptr, stream, false,
                    x, ldx);
}

q4k_status q4k_gemm_swiglu(const void* packed_pair, int64_t n, int64_t k, int act, const void* x_or_q8,
                           const void* da_f16, const void* ssum, int64_t m, int64_t ldx, void* h_ws,
                           size_t h_ws_bytes, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (n <= 0 || n % 256 || n >= kMaxDim / 2) return Q4K_ERR_SHAPE;   // n is the down projection's k
    q4k_status st = check_gemm_shape(2 * n, k, m);
    if (st != Q4K_OK) return st;
    if (!packed_pair) return Q4K_ERR_INVALID_ARG;
    if (act != Q4K_ACT_F32 && act != Q4K_ACT_Q8) return Q4K_ERR_INVALID_ARG;
    if (!aligned(packed_pair, 256)) return Q4K_ERR_ALIGNMENT;
    if (m == 0) return Q4K_OK;
    if (!h_ws) return Q4K_ERR_INVALID_ARG;
    if (!aligned(h_ws, 256)) return Q4K_ERR_ALIGNMENT;
    if (h_ws_bytes < static_cast<size_t>(ActLayout(m, n).total)) return Q4K_ERR_WORKSPACE;
    if (act == Q4K_ACT_F32) {
        st = q4k_act_quantize(static_cast<const float*>(x_or_q8), m, k, ldx, workspace, workspace_bytes, stream);
    } else {
        st = q4k_act_from_q8(static_cast<const int8_t*>(x_or_q8), static_cast<const uint16_t*>(da_f16),
                             static_cast<const int16_t*>(ssum), m, k, ldx, workspace, workspace_bytes, stream);
    }
    if (st != Q4K_OK) return st;
    return run_gemm(packed_pair, 2 * n, k, workspace, workspace_bytes, m, nullptr, Q4K_OUT_F32, 2 * n, nullptr, h_ws,
                    stream);
}

q4k_status q4k_gemm_swiglu_quantized(const void* packed_pair, int64_t n, int64_t k, void* workspace,
                                     size_t workspace_bytes, int64_t m, void* h_ws, size_t h_ws_bytes,
                                     cudaStream_t stream) {
    if (n <= 0 || n % 256 || n >= kMaxDim / 2) return Q4K_ERR_SHAPE;
    q4k_status st = check_gemm_shape(2 * n, k, m);
    if (st != Q4K_OK) return st;
    if (m == 0) return Q4K_OK;
    if (!h_ws) return Q4K_ERR_INVALID_ARG;
    if (!aligned(h_ws, 256)) return Q4K_ERR_ALIGNMENT;
    if (h_ws_bytes < static_cast<size_t>(ActLayout(m, n).total)) return Q4K_ERR_WORKSPACE;
    return run_gemm(packed_pair, 2 * n, k, workspace, workspace_bytes, m, nullptr, Q4K_OUT_F32, 2 * n, nullptr, h_ws,
                    stream);
}

size_t q6k_packed_bytes(int64_t n, int64_t k) {
    if (n <= 0 || k <= 0 || n % kTileN || k % 256 || n >= kMaxDim || k >= kMaxDim) return 0;
    return static_cast<size_t>(Q6Layout(n, k).total);
}

q4k_status q6k_pack_weights(const void* blocks, int64_t n, int64_t k, void* packed, size_t packed_bytes,
                            cudaStream_t stream) {
    if (n <= 0 || k <= 0 || n % kTileN || k % 256 || n >= kMaxDim || k >= kMaxDim) return Q4K_ERR_SHAPE;
    if (!blocks || !packed) return Q4K_ERR_INVALID_ARG;
    if (!aligned(packed, 256)) return Q4K_ERR_ALIGNMENT;
    if (packed_bytes < q6k_packed_bytes(n, k)) return Q4K_ERR_WORKSPACE;
    DeviceInfo* dev = nullptr;
    q4k_status st = device_info(&dev);
    if (st != Q4K_OK) return st;
    return from_cuda(launch_pack_q6k(static_cast<const uint8_t*>(blocks), n, k, static_cast<uint8_t*>(packed), stream));
}

q4k_status q6k_gemm(const void* packed_w, int64_t n, int64_t k, int act, const void* x_or_q8, const void* da_f16,
                    const void* ssum, int64_t m, int64_t ldx, void* y, int out_dtype, int64_t ldy, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream) {
    q4k_status st = check_gemm_shape(n, k, m);
    if (st != Q4K_OK) return st;
    if ((st = check_output(y, m, n, out_dtype, ldy)) != Q4K_OK) return st;
    if (!packed_w) return Q4K_ERR_INVALID_ARG;
    if (act != Q4K_ACT_F32 && act != Q4K_ACT_Q8) return Q4K_ERR_INVALID_ARG;
    if (!aligned(packed_w, 256)) return Q4K_ERR_ALIGNMENT;
    if (m == 0) return Q4K_OK;
    DeviceInfo* dev = nullptr;
    if (m > Q4K_SMALL_M || !gemv_q6k_fits(static_cast<int>(m), k)) {   // the tensor-core GEMM
        if (!workspace) return Q4K_ERR_INVALID_ARG;
        if (!aligned(workspace, 256)) return Q4K_ERR_ALIGNMENT;
        if (workspace_bytes < q4k_act_workspace_bytes(m, k)) return Q4K_ERR_WORKSPACE;
        if ((st = device_info(&dev)) != Q4K_OK) return st;
        if (act == Q4K_ACT_F32) {
            const float* xf = static_cast<const float*>(x_or_q8);
            if ((st = check_act_f32(xf, m, k, ldx)) != Q4K_OK) return st;
            st = from_cuda(launch_act_quantize(xf, m, k, ldx, workspace, stream));
        } else {
            const int8_t* q8 = static_cast<const int8_t*>(x_or_q8);
            if (!q8 || !da_f16 || !ssum) return Q4K_ERR_INVALID_ARG;
            if (ldx < k) return Q4K_ERR_SHAPE;
            if (!aligned(q8, 4) || ldx % 4 || !aligned(da_f16, 2) || !aligned(ssum, 2)) return Q4K_ERR_ALIGNMENT;
            st = from_cuda(launch_act_from_q8(q8, static_cast<const uint16_t*>(da_f16),
                                              static_cast<const int16_t*>(ssum), m, k, ldx, workspace, stream));
        }
        if (st != Q4K_OK) return st;
        return run_gemm(packed_w, n, k, workspace, workspace_bytes, m, y, out_dtype, ldy, nullptr, nullptr, stream,
                        true);
    }
    if ((st = device_info(&dev)) != Q4K_OK) return st;
    const Q6Layout W(n, k);
    const uint8_t* wb = static_cast<const uint8_t*>(packed_w);
    GemvParams g;
    std::memset(&g, 0, sizeof(g));
    g.nib = wb + W.lo;
    g.q6hi = wb + W.hi;
    g.sc = wb + W.sc;
    g.dsb = reinterpret_cast<const float*>(wb + W.dsb);
    g.q6 = 1;
    g.y = y;
    g.ldy = ldy;
    g.m = static_cast<int>(m);
    g.n = static_cast<int>(n);
    g.k = static_cast<int>(k);
    g.kc = static_cast<int>(k / 32);
    g.ksb = static_cast<int>(k / 256);
    g.out_bf16 = out_dtype == Q4K_OUT_BF16 ? 1 : 0;
    if (act == Q4K_ACT_F32) {
        const float* xf = static_cast<const float*>(x_or_q8);
        if ((st = check_act_f32(xf, m, k, ldx)) != Q4K_OK) return st;
        if (m <= kFusedQuantMaxM) {   // one launch: the kernel quantizes the activations itself
            g.xf = xf;
            g.ldx = ldx;
            return from_cuda(launch_gemv_q6k(g, stream));
        }
        const SmallMLayout L(m, k);
        if (!workspace) return Q4K_ERR_INVALID_ARG;
        if (!aligned(workspace, 256)) return Q4K_ERR_ALIGNMENT;
        if (workspace_bytes < static_cast<size_t>(L.total)) return Q4K_ERR_WORKSPACE;
        uint8_t* wsb = static_cast<uint8_t*>(workspace);
        int8_t* q8 = reinterpret_cast<int8_t*>(wsb + L.q8);
        uint16_t* da = reinterpret_cast<uint16_t*>(wsb + L.da);
        int16_t* ss = reinterpret_cast<int16_t*>(wsb + L.ssum);
        if ((st = q8_quantize_rows(xf, m, k, ldx, q8, da, ss, stream)) != Q4K_OK) return st;
        g.q8 = q8;
        g.da = da;
        g.ssum = ss;
        g.ldq = k;
        return from_cuda(launch_gemv_q6k(g, stream));
    }
    const int8_t* q8 = static_cast<const int8_t*>(x_or_q8);
    if (!q8 || !da_f16 || !ssum) return Q4K_ERR_INVALID_ARG;
    if (ldx < k) return Q4K_ERR_SHAPE;
    if (!aligned(q8, 16) || ldx % 16 || !aligned(da_f16, 16) || !aligned(ssum, 16)) return Q4K_ERR_ALIGNMENT;
    g.q8 = q8;
    g.da = static_cast<const uint16_t*>(da_f16);
    g.ssum = static_cast<const int16_t*>(ssum);
    g.ldq = ldx;
    return from_cuda(launch_gemv_q6k(g, stream));
}

unsigned int q4k_device_error_word(int reset) {
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != Q4K_OK) return 0xFFFFFFFFu;
    if (cudaDeviceSynchronize() != cudaSuccess) return 0xFFFFFFFFu;
    unsigned v = 0;
    if (cudaMemcpy(&v, dev->err_word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return 0xFFFFFFFFu;
    if (reset) {
        const unsigned z = 0;
        if (cudaMemcpy(dev->err_word, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return 0xFFFFFFFFu;
    }
    return v;
}

q4k_status q4k_device_status(int reset) {
    const unsigned v = q4k_device_error_word(reset);
    if (v == 0) return Q4K_OK;
    if (v == 0xFFFFFFFFu) return Q4K_ERR_CUDA;
    if ((v & 0xF00u) == 0x100u) return Q4K_ERR_TIMEOUT;
    return Q4K_ERR_CUDA;
}

q4k_status q4k_selftest_wait_timeout(int64_t timeout_ns, cudaStream_t stream) {
    if (timeout_ns < 1000 || timeout_ns > 10000000000LL) return Q4K_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    q4k_status st = device_info(&dev);
    if (st != Q4K_OK) return st;
    if (q4k_device_error_word(1) == 0xFFFFFFFFu) return Q4K_ERR_CUDA;
    if (launch_selftest_wait(dev->err_word, static_cast<uint64_t>(timeout_ns) * kCyclesPerNs, stream) != cudaSuccess)
        return Q4K_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return Q4K_ERR_CUDA;
    return q4k_device_status(1);
}

q4k_status q4k_peak_mma_s8(int64_t blocks, int64_t iters, int* sink, cudaStream_t stream) {
    if (blocks < 1 || blocks > (int64_t(1) << 20) || iters < 1 || iters > (int64_t(1) << 24)) return Q4K_ERR_INVALID_ARG;
    if (!sink) return Q4K_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    const q4k_status st = device_info(&dev);
    if (st != Q4K_OK) return st;
    return from_cuda(launch_peak_s8(blocks, iters, sink, stream));
}

q4k_status q4k_gemm_debug_chunk_acc(const void* packed_w, int64_t n, int64_t k, void* workspace,
                                    size_t workspace_bytes, int64_t m, float* y, int64_t ldy, float* chunk_acc,
                                    cudaStream_t stream) {
    if (!chunk_acc) return Q4K_ERR_INVALID_ARG;
    if (m < 0 || n <= 0 || k <= 0 || m * n * (k / 32) > (int64_t(1) << 26)) return Q4K_ERR_SHAPE;
    return run_gemm(packed_w, n, k, workspace, workspace_bytes, m, y, Q4K_OUT_F32, ldy, chunk_acc, nullptr, stream);
}

q4k_status q6k_gemm_debug_chunk_acc(const void* packed_w, int64_t n, int64_t k, void* workspace,
                                    size_t workspace_bytes, int64_t m, float* y, int64_t ldy, float* chunk_acc,
                                    cudaStream_t stream) {
    if (!chunk_acc) return Q4K_ERR_INVALID_ARG;
    if (m < 0 || n <= 0 || k <= 0 || m * n * (k / 32) > (int64_t(1) << 26)) return Q4K_ERR_SHAPE;
    return run_gemm(packed_w, n, k, workspace, workspace_bytes, m, y, Q4K_OUT_F32, ldy, chunk_acc, nullptr, stream,
                    true);
}

}  // extern "C"

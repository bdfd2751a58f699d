// q4k_gemm_static_workspace: the fused q4k_gemm with its activation
// workspace taken from a fixed array in the library's own device memory
// instead of a caller-supplied buffer.
//
// Who needs it: a caller that holds only its input and output pointers and
// has no device allocator to draw scratch from (a plain C host, or an engine
// whose memory is carved up once at start-up and that may not call
// cudaMalloc later, because cudaMalloc can synchronise the device and stall
// work already queued).  This entry point calls no cudaMalloc, cudaFree or
// any other allocating routine.
//
// The array lives for as long as the library stays loaded, one copy per
// device context (each device's primary context, for runtime-API callers).
// Every call in a context uses the same copy, so two calls that overlap in
// time on one device (different streams, or different host threads) race on
// it and corrupt each other's results: the caller must order them.  Nothing in the array needs to start at zero: the
// quantization step of each call rewrites every byte the GEMM step reads.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/q4k.h"

namespace q4k {
namespace {

constexpr size_t kStaticWsBytes = Q4K_STATIC_WORKSPACE_BYTES;

// The scratch array.  Host code must not use this name as a device address;
// the address comes from cudaGetSymbolAddress in static_ws_address below.
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

// The array's address in the current context, looked up on every call (the
// lookup allocates nothing).  A cached address could belong to a context that
// was since destroyed (cudaDeviceReset) or to another context on the same
// device (driver-API contexts), so none is kept.  The first lookup in a
// context loads this library's device code into it; that first call should
// therefore come before any stream capture.
q4k_status static_ws_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4K_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return Q4K_ERR_CUDA;
    if (major != 10 || minor != 3) return Q4K_ERR_UNSUPPORTED_DEVICE;   // the array exists in sm_103a code only
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || !ptr) return Q4K_ERR_CUDA;
    *out = ptr;
    return Q4K_OK;
}

}  // namespace
}  // namespace q4k

extern "C" {

size_t q4k_static_workspace_bytes(void) { return q4k::kStaticWsBytes; }

q4k_status q4k_gemm_static_workspace(const void* packed_w, int64_t n, int64_t k, int act, const void* x_or_q8,
                                     const void* da_f16, const void* ssum, int64_t m, int64_t ldx, void* y,
                                     int out_dtype, int64_t ldy, cudaStream_t stream) {
    if (act != Q4K_ACT_F32 && act != Q4K_ACT_Q8) return Q4K_ERR_INVALID_ARG;
    const size_t need = q4k_gemm_workspace_bytes(m, n, k, act);
    if (need == 0) return Q4K_ERR_SHAPE;
    if (need > q4k::kStaticWsBytes) return Q4K_ERR_WORKSPACE;   // m * k beyond the array
    void* ws = nullptr;
    const q4k_status st = q4k::static_ws_address(&ws);
    if (st != Q4K_OK) return st;
    return q4k_gemm(packed_w, n, k, act, x_or_q8, da_f16, ssum, m, ldx, y, out_dtype, ldy, ws, q4k::kStaticWsBytes,
                    stream);
}

}  // extern "C"

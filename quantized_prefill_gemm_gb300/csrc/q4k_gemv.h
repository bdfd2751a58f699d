// The small-M (decode-sized) products' parameters and launchers (gemv.cu,
// gemv_stream.cu), apart from the tensor-core GEMM's declarations.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace q4k {

// Small-M product (gemv.cu): packed weights as for the GEMM, activations as
// the q8 SoA of q8_quantize_rows (q8 rows, d_a and ssum 16-byte aligned,
// ldq % 16 == 0).
struct GemvParams {
    const uint8_t* nib;      // packed quants  [nt][kc][128][16 B]
    const uint8_t* sc;       // packed scales  [nt][kc][128]
    const uint8_t* mq;       // packed mins    [nt][kc][128]
    const float* dsb;        // super-block d    [nt][ksb][128]
    const float* dmn;        // super-block dmin [nt][ksb][128]
    const int8_t* q8;        // [m][ldq]
    const uint16_t* da;      // f16 bits [m][kc]
    const int16_t* ssum;     // [m][kc]
    const float* xf;         // fp32 activations [m][ldx]; when set, quantized in the kernel (q8/da/ssum unused)
    // Q6_K weights (Q6Layout) instead of Q4_K: nib = lo, sc = the i8 scale
    // pairs, dsb = d; mq and dmn unused
    const uint8_t* q6hi;
    int q6;
    void* y;                 // [m][ldy]
    int64_t ldq, ldx, ldy;
    int m, n, k, kc, ksb;
    int out_bf16;
};

cudaError_t launch_gemv(const GemvParams& p, cudaStream_t s);
// The streamed small-M form (m <= 4, Q4_K or Q6_K by p.q6); leaves *launched
// false, launching nothing, when the call is outside its range or its shared
// memory would not fit.
cudaError_t launch_gemv_stream(const GemvParams& p, cudaStream_t s, bool* launched);
// Q6_K small-M product (p.q6 set); gemv_q6k_fits says whether m tokens of k
// activations fit its shared memory
bool gemv_q6k_fits(int m, int64_t k);
cudaError_t launch_gemv_q6k(const GemvParams& p, cudaStream_t s);

}  // namespace q4k

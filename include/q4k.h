/*
 * q4k.h -- C ABI of the Q4_K x q8 prefill GEMM for NVIDIA GB300 (sm_103a).
 *
 * The operation (all page references are to the yusiwen.cn minfer
 * "cuda_optimization_steps" pages):
 *
 *   Y[t, o] = sum_k W[o, k] * X[t, k]
 *
 * W is stored in Q4_K super-blocks (256 weights: f16 d and dmin, eight 32-weight
 * sub-blocks with 6-bit scale sc and 6-bit min m, 4-bit quants q; w = d*sc*q -
 * dmin*m).  X is quantized into 32-element q8 blocks, each with an f16 scale
 * d_a and the i16 sum ssum of its q8 values ("34 · r31 — q-major sda
 * scale-read repack", §1 Background).  Each 32-k chunk is reduced as an exact
 * integer dot product and rescaled by the two-term rank-1 rescale
 *   d_a*(d*sc)*sum(q*qa) + d_a*ssum*(-dmin*m)
 * ("34 · r31", §1-§2: the A-side pair (d_a, ssum) and the B-side pair
 * (d*sc, -dmin*m); "22 · r17 — Wide warp remap", §1: the r15 rank-1 fold).
 *
 * Conventions for every entry point
 *   - Pointers named as device memory are device memory owned by the caller.
 *     The library never allocates, frees or synchronises on these calls
 *     (the diagnostics at the end of this header are the documented
 *     exceptions: they synchronise).
 *   - Every call is asynchronous on `stream` (0 = the legacy default stream).
 *     The returned status covers argument validation and launch errors;
 *     faults inside a kernel surface at the caller's next synchronisation.
 *     Internal waits of the GEMM are bounded: on a timeout the kernel records
 *     an error word (see q4k_device_status) and returns instead of hanging.
 *   - Matrices are row-major; leading dimensions are in elements.
 *   - No C++ exception crosses this boundary.
 */
#ifndef Q4K_H
#define Q4K_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cudaStream_t;   /* same type as the CUDA runtime's */

typedef enum q4k_status {
    Q4K_OK = 0,
    Q4K_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum  */
    Q4K_ERR_SHAPE = 2,              /* k % 256, n % 128, ld < row length ...  */
    Q4K_ERR_ALIGNMENT = 3,          /* pointer or leading dimension alignment */
    Q4K_ERR_WORKSPACE = 4,          /* workspace / packed buffer too small    */
    Q4K_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not sm_103           */
    Q4K_ERR_CUDA = 6,               /* a CUDA runtime / driver call failed    */
    Q4K_ERR_TIMEOUT = 7             /* a bounded device-side wait ran out     */
} q4k_status;

typedef enum q4k_act_kind {
    Q4K_ACT_F32 = 0,   /* x is fp32 [m][ldx]; quantized inside q4k_gemm      */
    Q4K_ACT_Q8 = 1     /* x is the q8 SoA of q8_quantize_rows (see there)    */
} q4k_act_kind;

typedef enum q4k_out_dtype {
    Q4K_OUT_F32 = 0,
    Q4K_OUT_BF16 = 1   /* fp32 result rounded to bf16, round-to-nearest-even */
} q4k_out_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* q4k_status_string(int status);

/* ABI version of this header (bumped on any incompatible change). */
#define Q4K_ABI_VERSION 1
int q4k_abi_version(void);

/* ------------------------------------------------------------------------
 * q8_quantize_rows -- activation quantization into 32-element q8 blocks.
 * ("34 · r31 — q-major sda scale-read repack", §1: each q8 block carries an
 * f16 scale d and an i16 ssum, the sum of its q8 values.)
 * Per block of 32 consecutive k of one token:
 *   amax = max|x|;  if amax < 2^-120: qa = 0, ssum = 0, d_a = +0;
 *   else d = RN32(amax/127), inv = RN32(127/amax),
 *        qa = clamp(rint_half_even(RN32(x*inv)), -127, 127),
 *        ssum = sum(qa), d_a = RN16(d).
 * Bit-exact by construction (IEEE fp32 ops in this order, no contraction).
 *   x       device, fp32 [m][ldx]; 16-byte aligned, ldx % 4 == 0, ldx >= k
 *   q8      device, int8 [m][k]   (4-byte aligned)
 *   da_f16  device, f16 bit patterns [m][k/32]
 *   ssum    device, int16 [m][k/32]
 *   k % 32 == 0; m == 0 is a no-op.  x must be finite.
 * ------------------------------------------------------------------------ */
q4k_status q8_quantize_rows(const float* x, int64_t m, int64_t k, int64_t ldx,
                            int8_t* q8, uint16_t* da_f16, int16_t* ssum,
                            cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Weight repack (load time, not on the per-token path).
 * q4k_blocks  device, [n][k/256] canonical 144-byte Q4_K blocks (16-byte
 *             aligned): bytes 0-1 d (f16), 2-3 dmin (f16), 4-15 the sixteen
 *             6-bit scales/mins, 16-143 the 4-bit quants (GGUF Q4_K order).
 * packed      device, q4k_packed_bytes(n, k) bytes (256-byte aligned); an
 *             opaque layout consumed only by q4k_gemm / q4k_gemm_quantized.
 * n % 128 == 0, k % 256 == 0.
 * ------------------------------------------------------------------------ */
size_t q4k_packed_bytes(int64_t n, int64_t k);
q4k_status q4k_pack_weights(const void* q4k_blocks, int64_t n, int64_t k,
                            void* packed, size_t packed_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * q4k_gemm -- Y = W * X^T with the per-32-k rescale (the path above).
 *   packed_w  from q4k_pack_weights(n, k)
 *   act == Q4K_ACT_F32: x_or_q8 = fp32 [m][ldx] (same rules as
 *                       q8_quantize_rows); da_f16 and ssum are ignored.
 *   act == Q4K_ACT_Q8 : x_or_q8 = int8 q8 [m][ldx] (ldx % 4 == 0, 4-byte
 *                       aligned), da_f16 = f16 bits [m][k/32],
 *                       ssum = int16 [m][k/32], as written by q8_quantize_rows.
 *   y         device, [m][ldy] fp32 (ldy % 4 == 0) or bf16 (ldy % 8 == 0),
 *             16-byte aligned; columns [n, ldy) are not touched.
 *   workspace device, >= q4k_gemm_workspace_bytes(m, n, k, act) bytes,
 *             256-byte aligned; contents are scratch, overwritten per call.
 * n % 128 == 0, k % 256 == 0, m >= 0.
 * Accuracy: per output, |y - y_exact| <= 1e-4 * sum_k |w_k * a_k| (fp32
 * output) where a = d_a*qa, and the per-chunk integer dot products are exact.
 * Small M: for 1 <= m <= Q4K_SMALL_M tokens (decode-sized batches) the call
 * runs a CUDA-core kernel whose cost is reading the packed weights (integer
 * dot products with dp4a, same rescale and accuracy contract).  With f32
 * input and m <= Q4K_FUSED_QUANT_M it is one launch that quantizes the
 * activations inside the kernel (the same q8, d_a and ssum bits as
 * q8_quantize_rows) and leaves `workspace` untouched (it may then be NULL);
 * for larger m the q8 SoA is first written to the start of `workspace`.  The
 * q8 path reads the caller's arrays directly when q8, da_f16 and ssum are
 * 16-byte aligned and ldx % 16 == 0 (otherwise it takes the general path).
 * ------------------------------------------------------------------------ */
#define Q4K_SMALL_M 16
#define Q4K_FUSED_QUANT_M 4
size_t q4k_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, int act);
q4k_status q4k_gemm(const void* packed_w, int64_t n, int64_t k,
                    int act, const void* x_or_q8, const void* da_f16, const void* ssum,
                    int64_t m, int64_t ldx,
                    void* y, int out_dtype, int64_t ldy,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * The two halves of q4k_gemm, for callers that multiply one quantized
 * activation by several weight matrices (e.g. q, k and v of one layer).
 * q4k_act_quantize   fp32 x [m][ldx] -> the GEMM operand form in `workspace`
 * q4k_act_from_q8    q8 SoA (as q8_quantize_rows writes it) -> same form
 * q4k_gemm_quantized workspace (filled by one of the two, same m and k) -> Y
 * workspace: >= q4k_act_workspace_bytes(m, k) bytes, 256-byte aligned.  The
 * operand part is only read by the GEMM and may feed any number of calls;
 * the GEMM also uses a scratch part of the workspace (about 10 MB, for the
 * partial tiles of the work it splits along k to balance the last wave over
 * the SMs), so GEMMs that may run at the same time (different streams) must
 * not share a workspace.
 * ------------------------------------------------------------------------ */
size_t q4k_act_workspace_bytes(int64_t m, int64_t k);
q4k_status q4k_act_quantize(const float* x, int64_t m, int64_t k, int64_t ldx,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);
q4k_status q4k_act_from_q8(const int8_t* q8, const uint16_t* da_f16, const int16_t* ssum,
                           int64_t m, int64_t k, int64_t ldq,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);
q4k_status q4k_gemm_quantized(const void* packed_w, int64_t n, int64_t k,
                              void* workspace, size_t workspace_bytes, int64_t m,
                              void* y, int out_dtype, int64_t ldy, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * q4k_gemm_inkernel_quant -- q4k_gemm for fp32 activations in one kernel
 * launch: the GEMM kernel quantizes x into `workspace` itself ("34 · r31 --
 * q-major sda scale-read repack", §1 for the q8 blocks; the same operation
 * order as q4k_act_quantize, so the operand bits are the same).  Its warps
 * with no other work at that moment quantize: the tiles the first wave of
 * output tiles reads before it starts, the rest while the tiles run; a
 * 128-token tile's product starts once every slice of it is quantized (the
 * CTAs wait for one another, so the kernel is a cooperative launch: it
 * fails with Q4K_ERR_CUDA rather than starting when the GPU cannot hold all
 * of its CTAs at once).  On a GB300 it measured 5-7% slower than q4k_gemm's
 * separate quantization pass (512 to 2630 tokens, 4096-11008 features),
 * which is why q4k_gemm does not take this path.
 *   packed_w, n, k, y, out_dtype, ldy: as q4k_gemm.
 *   x [m][ldx] fp32, 16-byte aligned, ldx % 4 == 0, ldx >= k; m >= 0 (the
 *   tensor-core GEMM for every m, no small-M path).
 *   workspace: >= q4k_act_workspace_bytes(m, k) bytes, 256-byte aligned; on
 *   return its operand part holds what q4k_act_quantize would write.  It also
 *   holds one 64-bit counter per 128-token tile, tagged with the call: the
 *   workspace needs no initialisation (a call never mistakes an earlier
 *   call's counts, or leftover bytes, for its own unless they happen to hold
 *   this call's 48-bit tag), and calls that may overlap in time must not
 *   share it.
 *   Output: identical bits to q4k_act_quantize + q4k_gemm_quantized except
 *   where the two split different output tiles along k to balance the last
 *   wave (this call orders the tiles output-tile first), where the fp32 sums
 *   are added in another order; the accuracy contract is q4k_gemm's.
 * ------------------------------------------------------------------------ */
q4k_status q4k_gemm_inkernel_quant(const void* packed_w, int64_t n, int64_t k, const float* x, int64_t m,
                                   int64_t ldx, void* y, int out_dtype, int64_t ldy,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Gate/up pair with a SiLU(gate)*up epilogue that produces the down
 * projection's quantized input.  The pages measure LLaMA-7B's linear layers
 * ("34 · r31 — q-major sda scale-read repack", Result: 7B q4_K whole-prefill);
 * its feed-forward block feeds the down projection h = SiLU(g) * u with
 * g = W_gate x, u = W_up x and SiLU(g) = g / (1 + e^-g).  Fusing it into the
 * gate/up product's epilogue removes the round trip of g and u through HBM
 * and the separate activation quantization of h.
 *
 * q4k_pack_swiglu_weights  gate and up Q4_K blocks ([n][k/256] x 144 B each,
 *            device, 16-byte aligned) -> one packed matrix of 2n rows in
 *            which each 128-row tile holds 64 outputs' gate and up rows;
 *            packed: q4k_swiglu_packed_bytes(n, k) bytes, 256-byte aligned.
 * q4k_gemm_swiglu  x (act and x_or_q8, da_f16, ssum, m, ldx as for q4k_gemm)
 *            times the pair; h_ws receives, for every token, the q8
 *            quantization of h (32-element blocks along n, the same rule as
 *            q8_quantize_rows) in the operand form of q4k_act_quantize for
 *            an m x n input: pass it to q4k_gemm_quantized with the down
 *            projection's weights (k = n).
 *            h_ws: >= q4k_act_workspace_bytes(m, n) bytes, 256-byte aligned;
 *            workspace: >= q4k_gemm_workspace_bytes(m, 2n, k, act), scratch
 *            for x's operand form; the two must not overlap.
 * h is evaluated in a fixed fp32 order, each step one IEEE round-to-nearest
 * operation.  With t = -g: SiLU = -0 if t > 80; SiLU = g if t < -87;
 * otherwise SiLU = RN(g * R(RN(1 + E(t)))); then h = RN(SiLU * u).
 * E(t) = RN(p(r) * 2^n) where n = rint_even(RN(t * RN32(log2 e))),
 * r = RN(RN(t - n*355/512) - RN(n*C2)), C2 = RN32(ln 2 - 355/512), and p is
 * the degree-7 Taylor polynomial of e^r in Horner form with fp32 coefficients
 * RN32(1/j!) (each step RN(RN(p*r) + c)).  R(s): y = the float with bits
 * 0x7EF311C2 - bits(s), then three times y = RN(y * RN(2 - RN(s * y))).
 * g and u are the fp32 values the same product writes with f32 output.
 * Packing needs n % 64 == 0; q4k_gemm_swiglu needs n % 256 == 0 (n is the
 * down projection's k), k % 256 == 0, m >= 0.
 * ------------------------------------------------------------------------ */
size_t q4k_swiglu_packed_bytes(int64_t n, int64_t k);
q4k_status q4k_pack_swiglu_weights(const void* gate_blocks, const void* up_blocks, int64_t n, int64_t k,
                                   void* packed, size_t packed_bytes, cudaStream_t stream);
q4k_status q4k_gemm_swiglu(const void* packed_pair, int64_t n, int64_t k,
                           int act, const void* x_or_q8, const void* da_f16, const void* ssum,
                           int64_t m, int64_t ldx, void* h_ws, size_t h_ws_bytes,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);
/* The second half of q4k_gemm_swiglu, for x already in operand form (from
 * q4k_act_quantize or q4k_act_from_q8 with the same m and k). */
q4k_status q4k_gemm_swiglu_quantized(const void* packed_pair, int64_t n, int64_t k,
                                     void* workspace, size_t workspace_bytes, int64_t m,
                                     void* h_ws, size_t h_ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Q6_K weights.  The series moves on from Q4_K to a Q6_K line
 * ("34 · r31 — q-major sda scale-read repack", §5 Results, post-hoc notes);
 * the pages give no layout for it.  Blocks follow the public GGUF Q6_K
 * format: 256 weights in 210 bytes (ql[128] low 4 bits, qh[64] high 2 bits,
 * sc[16] signed 8-bit scales of 16 weights each, d f16 at bytes 208-209),
 * w = d * sc * (q - 32).
 * q6k_pack_weights  blocks [n][k/256] x 210 B (device) -> packed
 *            (q6k_packed_bytes(n, k) bytes, 256-byte aligned).
 * q6k_gemm   as q4k_gemm (same arguments, activation forms and accuracy
 *            contract): per 32-k block the exact integer
 *            sum_s sc_s * sum (q - 32) * qa (two 16-weight sub-blocks), then
 *            d_a * d times it.  For 1 <= m <= Q4K_SMALL_M tokens whose
 *            activations fit the small-M kernel's shared memory (m x k bytes
 *            plus scales, at most ~200 KB) it runs on the CUDA cores: with
 *            f32 input and m <= Q4K_FUSED_QUANT_M the kernel quantizes the
 *            activations itself (workspace unused), otherwise the q8 SoA goes
 *            to the start of `workspace`.  Larger m take the tensor-core
 *            GEMM, which quantizes into `workspace` as q4k_gemm does.
 *            workspace_bytes >= q4k_gemm_workspace_bytes(m, n, k, act).
 * n % 128 == 0, k % 256 == 0.
 * ------------------------------------------------------------------------ */
size_t q6k_packed_bytes(int64_t n, int64_t k);
q4k_status q6k_pack_weights(const void* q6k_blocks, int64_t n, int64_t k,
                            void* packed, size_t packed_bytes, cudaStream_t stream);
q4k_status q6k_gemm(const void* packed_w, int64_t n, int64_t k,
                    int act, const void* x_or_q8, const void* da_f16, const void* ssum,
                    int64_t m, int64_t ldx,
                    void* y, int out_dtype, int64_t ldy,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * q4k_gemm_static_workspace -- q4k_gemm without a workspace argument.
 * Library addition with no counterpart in the pages: it exists for callers
 * that cannot hand the library scratch memory, e.g. a plain C host that holds
 * only its input and output pointers, or an engine that carves its device
 * memory once at start-up and must not call cudaMalloc afterwards (cudaMalloc
 * can synchronise the device).  It allocates nothing: the activation
 * workspace is a fixed array of Q4K_STATIC_WORKSPACE_BYTES in the library's
 * own device memory (one per device context, alive while the library is
 * loaded).
 *   Arguments, layouts and results: as q4k_gemm (same kernels, so the output
 *   is identical to q4k_gemm's on the same inputs).
 *   Limit: q4k_gemm_workspace_bytes(m, n, k, act) must not exceed
 *   Q4K_STATIC_WORKSPACE_BYTES (64 MiB: e.g. m = 2048 tokens at k = 11008);
 *   larger problems return Q4K_ERR_WORKSPACE before anything is launched.
 *   Set-up: every call looks up the array's address in the current
 *   context (cudaGetSymbolAddress, with the device current; nothing is
 *   cached, so a reset device or another context never sees a stale
 *   address).  The first lookup in a context loads the library's device code
 *   into it: make the first call on each device before any stream capture.
 *   Sharing: all calls on one device use the same array and leave the last
 *   call's contents in it.  Calls that overlap in time on one device (other
 *   streams, other host threads) race on it; the caller must order them.
 *   Nothing in it needs clearing: each call rewrites what it reads.
 * q4k_static_workspace_bytes returns Q4K_STATIC_WORKSPACE_BYTES.
 * ------------------------------------------------------------------------ */
#define Q4K_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)
size_t q4k_static_workspace_bytes(void);
q4k_status q4k_gemm_static_workspace(const void* packed_w, int64_t n, int64_t k,
                                     int act, const void* x_or_q8, const void* da_f16,
                                     const void* ssum, int64_t m, int64_t ldx,
                                     void* y, int out_dtype, int64_t ldy, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostics (these synchronise the current device).
 * q4k_device_error_word  raw device-side error word of the current device
 *                        (0 = none; 0x1XX = a bounded wait ran out at site XX);
 *                        reset != 0 clears it.
 * q4k_device_status      the same, mapped to a q4k_status.
 * q4k_selftest_wait_timeout  launches one CTA that waits on a barrier nothing
 *                        will complete, with the given limit (ns, 1e3..1e10),
 *                        and returns the status the host reads back: it must
 *                        be Q4K_ERR_TIMEOUT.  Exercises the bounded-wait path
 *                        without faulting or hanging the GPU.
 * q4k_peak_mma_s8        diagnostics for the roofline, not part of the product:
 *                        launches `blocks` CTAs of 256 threads whose warps
 *                        each issue iters x 8 dense mma.sync m16n8k32 s8 x s8
 *                        -> s32 on register operands and nothing else (sm_103a
 *                        has no integer tcgen05 MMA, so this is the GPU's INT8
 *                        tensor rate); sink (device, >= blocks ints) receives
 *                        one checksum per CTA.  The caller times the launch:
 *                        blocks * 8 * iters * 8 * 8192 integer ops.
 *                        Asynchronous; INVALID_ARG outside 1 <= blocks <= 2^20,
 *                        1 <= iters <= 2^24 or for a null sink.
 * q4k_gemm_debug_chunk_acc  q4k_gemm_quantized with fp32 output that also
 *                        writes every per-chunk accumulator J[t][o][c] =
 *                        sum_{k in chunk c} (sc*q)[o,k]*qa[t,k] (exact
 *                        integers) to chunk_acc [m][n][k/32]; test hook,
 *                        limited to m*n*(k/32) <= 2^26.  Asynchronous.
 * q6k_gemm_debug_chunk_acc  the same for Q6_K weights on the tensor-core
 *                        path: J[t][o][c] = sum_s sc_s * sum (q - 32) * qa
 *                        over the chunk's two sub-blocks; workspace holds the
 *                        operand form (from q6k_gemm's own quantization, i.e.
 *                        a prior q6k_gemm call with m > 16 on it, or
 *                        q4k_act_quantize).
 * ------------------------------------------------------------------------ */
unsigned int q4k_device_error_word(int reset);
q4k_status q4k_device_status(int reset);
q4k_status q4k_selftest_wait_timeout(int64_t timeout_ns, cudaStream_t stream);
q4k_status q4k_peak_mma_s8(int64_t blocks, int64_t iters, int* sink, cudaStream_t stream);
q4k_status q4k_gemm_debug_chunk_acc(const void* packed_w, int64_t n, int64_t k,
                                    void* workspace, size_t workspace_bytes, int64_t m,
                                    float* y, int64_t ldy, float* chunk_acc, cudaStream_t stream);
q4k_status q6k_gemm_debug_chunk_acc(const void* packed_w, int64_t n, int64_t k,
                                    void* workspace, size_t workspace_bytes, int64_t m,
                                    float* y, int64_t ldy, float* chunk_acc, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* Q4K_H */

"""q4k_gemm for decode-sized batches (1 <= m <= 16 tokens): the CUDA-core
small-M paths (the streamed kernel: dp4a for m <= 4, integer mma.sync for
5 <= m <= 16 of q8 input when the staged activations fit; the register-held
kernels otherwise), compared with the oracle.

Same bar as the GEMM: per element |y_gpu - y_oracle| <= 1e-4 * sum_k |w_k a_k|
(plus one bf16 rounding for bf16 output).  The shapes span one and several
128-row tiles, super-block counts that fill no whole number of the kernels'
stages or shares (k = 11008 has 43), several row groups per CTA, every token
count class (1, 2, 3-4, 5-8, 9-16), both activation forms, and q8 arrays the
path cannot take directly (it then uses the general path).
"""
import numpy as np
import pytest
import torch

from tests.gpu_common import DEV, assert_close, make_case, oracle_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4k():
    from quantized_prefill_gemm_gb300 import q4k as mod

    mod.q4k_device_error_word(reset=True)
    yield mod
    assert mod.q4k_device_error_word() == 0


def _check(q4k, n, k, m, kind, seed, out="f32", act="f32"):
    blocks, x = make_case(n, k, m, kind, seed)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    if act == "q8":
        q, da, ss = q4k.q8_quantize_rows(to_dev(x))
        y = q4k.q4k_gemm(packed, n, k, q, out_dtype=out, da=da, ssum=ss)
    else:
        y = q4k.q4k_gemm(packed, n, k, to_dev(x), out_dtype=out)
    torch.cuda.synchronize()
    got = y.float().cpu().double().numpy()
    want, scale = oracle_rows(blocks, x, np.arange(m))
    return assert_close(got, want, scale, out, f"small-M {m}x{n}x{k} {act} {out}")


@pytest.mark.parametrize("m", [1, 2, 3, 5, 8, 13, 16])
def test_token_counts(q4k, m):
    _check(q4k, 256, 512, m, "normal", 20 + m)


@pytest.mark.parametrize("m", [1, 7, 16])
def test_q8_input(q4k, m):
    _check(q4k, 384, 768, m, "outlier", 40 + m, act="q8")


def test_q8_input_unaligned_rows_take_general_path(q4k):
    """q8 rows 4-byte aligned only (ldx = k + 4): still correct."""
    n, k, m = 256, 512, 4
    blocks, x = make_case(n, k, m, "normal", 50)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    q, da, ss = q4k.q8_quantize_rows(to_dev(x))
    qw = torch.zeros((m, k + 4), dtype=torch.int8, device=DEV)
    qw[:, :k] = q
    y = q4k.q4k_gemm(packed, n, k, qw[:, :k], out_dtype="f32", da=da, ssum=ss)
    torch.cuda.synchronize()
    want, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(y.cpu().double().numpy(), want, scale, "f32", "unaligned q8")


@pytest.mark.parametrize("n,k,m,out", [(4096, 4096, 1, "bf16"), (4096, 11008, 8, "bf16"),
                                       (11008, 4096, 16, "f32"), (256, 14336, 16, "f32")])
def test_decode_sizes(q4k, n, k, m, out):
    """The 7B projections at decode batch sizes, every output checked (the
    last shape's 16 x 14336 activations do not fit the persistent form's
    shared memory: it takes the per-group form)."""
    _check(q4k, n, k, m, "silu_mul" if k >= 11008 else "normal", 60 + m, out=out)


@pytest.mark.parametrize("n,k,m,out", [(4096, 11008, 1, "bf16"), (12288, 4096, 1, "bf16"),
                                       (22016, 4096, 1, "bf16"), (128, 256, 2, "f32"), (640, 2304, 3, "f32"),
                                       (640, 2304, 6, "f32"), (4096, 11008, 16, "bf16"), (512, 11008, 12, "f32")])
def test_streamed_shapes(q4k, n, k, m, out):
    """Shapes that exercise the streamed kernel in particular, every output
    checked: the 7B down projection (43 super-blocks, so each group ends with
    a stage of 3), q|k|v and gate|up stored as one matrix (768 and 1376
    16-row groups: several per CTA), a single super-block (a one-super-block
    stage), 40 groups with 9 super-blocks (a short second stage), and the
    tensor-core form with 6 tokens and with 12 and 16 tokens of k = 11008
    (too many staged activations for one pass: two passes of 8 tokens)."""
    _check(q4k, n, k, m, "silu_mul" if k >= 11008 else "normal", 90 + m, out=out)


def test_streamed_repeats_bitwise(q4k):
    """Two calls of the streamed kernel give identical bits (each row is summed
    in one CTA in a fixed order), for fp32 and for q8 input."""
    n, k, m = 4096, 4096, 1
    blocks, x = make_case(n, k, m, "normal", 95)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    xd = to_dev(x)
    q, da, ss = q4k.q8_quantize_rows(xd)
    a = q4k.q4k_gemm(packed, n, k, xd, out_dtype="bf16")
    b = q4k.q4k_gemm(packed, n, k, xd, out_dtype="bf16")
    c = q4k.q4k_gemm(packed, n, k, q, out_dtype="bf16", da=da, ssum=ss)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


def test_matches_general_path_and_repeats(q4k):
    """Small-M result vs the tensor-core path on the same quantized input, and
    two calls give identical bits (the 16 partial sums are added in a fixed order)."""
    n, k, m = 512, 1024, 9
    blocks, x = make_case(n, k, m, "normal", 70)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    xd = to_dev(x)
    y1 = q4k.q4k_gemm(packed, n, k, xd, out_dtype="f32")
    y2 = q4k.q4k_gemm(packed, n, k, xd, out_dtype="f32")
    ws = q4k.q4k_act_quantize(xd)
    yg = q4k.q4k_gemm_quantized(packed, n, k, ws, m, "f32")
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    _, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(y1.cpu().double().numpy(), yg.cpu().double().numpy(), scale, "f32", "small-M vs GEMM")


def _special_blocks(x):
    """Overwrite some 32-element blocks with the quantizer's special cases:
    all zero, below the 2^-120 zero-block threshold, subnormal, a single
    non-zero element, an amax just above the threshold, halves that round to
    even (x * 127 / amax = j + 0.5), and all-negative."""
    x = x.copy()
    m, k = x.shape
    kc = k // 32
    for t in range(m):
        c = (3 * t) % kc
        x[t, 32 * c:32 * c + 32] = 0.0
        c = (3 * t + 1) % kc
        x[t, 32 * c:32 * c + 32] = np.float32(1e-37) * np.sign(x[t, 32 * c:32 * c + 32])
        c = (3 * t + 2) % kc
        x[t, 32 * c:32 * c + 32] = np.float32(1e-40)
        c = (13 * t + 17) % kc
        x[t, 32 * c:32 * c + 32] *= np.float32(2e-36) / np.abs(x[t, 32 * c:32 * c + 32]).max()   # just live
        c = (5 * t + 7) % kc
        x[t, 32 * c:32 * c + 32] = 0.0
        x[t, 32 * c + 5] = -3.0
        c = (7 * t + 11) % kc
        x[t, 32 * c:32 * c + 32] = (np.arange(32, dtype=np.float32) + 0.5) * np.float32(1.0 / 127.0)
        x[t, 32 * c + 31] = 1.0   # amax 1: x * 127 = j + 0.5 for the other 31
        c = (11 * t + 13) % kc
        x[t, 32 * c:32 * c + 32] = -np.abs(x[t, 32 * c:32 * c + 32]) - np.float32(0.25)
    return x


@pytest.mark.parametrize("n,k,m,kind", [(256, 512, 1, "normal"), (384, 768, 3, "outlier"),
                                        (512, 11008, 4, "silu_mul"), (256, 4096, 2, "special"),
                                        (256, 4096, 4, "special"), (128, 2816, 1, "special")])
def test_in_kernel_quantization_matches_prepass_bits(q4k, n, k, m, kind):
    """fp32 activations (up to 4 tokens) are quantized inside the small-M kernel.  The q8, d_a
    and ssum it stages must be the stand-alone quantizer's bit for bit, so the
    output equals, bit for bit, the same kernel fed the quantizer's arrays;
    both are also checked against the oracle."""
    blocks, x = make_case(n, k, m, "normal" if kind == "special" else kind, 80 + m)
    if kind == "special":
        x = _special_blocks(x)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    xd = to_dev(x)
    y_fused = q4k.q4k_gemm(packed, n, k, xd, out_dtype="f32")
    q, da, ss = q4k.q8_quantize_rows(xd)
    y_pre = q4k.q4k_gemm(packed, n, k, q, out_dtype="f32", da=da, ssum=ss)
    torch.cuda.synchronize()
    assert torch.equal(y_fused, y_pre)
    want, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(y_fused.cpu().double().numpy(), want, scale, "f32", f"in-kernel quantization {kind}")


def test_in_kernel_quantization_strided_rows_and_no_workspace(q4k):
    """Row stride ldx > k, and the fp32 small-M call made with a NULL
    workspace (it does not use one)."""
    import ctypes

    n, k, m = 256, 1024, 3
    blocks, x = make_case(n, k, m, "outlier", 90)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    xw = torch.zeros((m, k + 12), dtype=torch.float32, device=DEV)
    xw[:, :k] = to_dev(x)
    y = torch.full((m, n), float("nan"), dtype=torch.float32, device=DEV)
    st = q4k.LIB.q4k_gemm(ctypes.c_void_p(packed.data_ptr()), n, k, q4k.ACT_F32, ctypes.c_void_p(xw.data_ptr()),
                          None, None, m, k + 12, ctypes.c_void_p(y.data_ptr()), 0, n, None, 0,
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, q4k.LIB.q4k_status_string(st)
    torch.cuda.synchronize()
    want, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(y.cpu().double().numpy(), want, scale, "f32", "strided fp32 rows, no workspace")


@pytest.mark.parametrize("m", [2, 8])
def test_long_k_takes_the_register_held_kernels(q4k, m):
    """k = 20480 with 8 tokens stages more activations than the streamed
    kernel holds: the register-held kernels take it (and m = 2 the streamed
    one); every output checked."""
    _check(q4k, 128, 20480, m, "normal", 130 + m, out="f32", act="q8")


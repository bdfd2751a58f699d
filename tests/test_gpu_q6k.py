"""q6k_gemm (Q6_K weights) on the GPU vs the oracle: the small-M path for
decode sizes and the tensor-core GEMM above them.

Bar as for Q4_K: per element |y_gpu - y_oracle| <= 1e-4 * sum_k |w_k * a_k|
(plus one bf16 rounding for bf16 output); fp32 activations quantized inside
the kernel must give the bits of the same kernel fed the quantizer's q8.
"""
import numpy as np
import pytest
import torch

from oracle import q6k_blocks as oq6
from oracle import q8 as oq8
from quantized_prefill_gemm_gb300 import inputs
from tests.gpu_common import DEV, assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4k():
    from quantized_prefill_gemm_gb300 import q4k as mod

    mod.q4k_device_error_word(reset=True)
    yield mod
    assert mod.q4k_device_error_word() == 0


def _oracle(blocks, x):
    f = oq6.decode(blocks)
    qa, da, _ = oq8.quantize_rows(x)
    return oq6.gemm_blockwise(f, qa, da), oq6.abs_scale(f, qa, da)


def _check(q4k, n, k, m, seed, out="f32", act="f32", kind="normal"):
    blocks = inputs.q6k_blocks(n, k, seed)
    x = inputs.activations(m, k, seed, kind)
    packed = q4k.q6k_pack_weights(to_dev(blocks), n, k)
    if act == "q8":
        q, da, ss = q4k.q8_quantize_rows(to_dev(x))
        y = q4k.q6k_gemm(packed, n, k, q, out_dtype=out, da=da, ssum=ss)
    else:
        y = q4k.q6k_gemm(packed, n, k, to_dev(x), out_dtype=out)
    torch.cuda.synchronize()
    want, scale = _oracle(blocks, x)
    assert_close(y.float().cpu().double().numpy(), want, scale, out, f"q6k {m}x{n}x{k} {act} {out}")


@pytest.mark.parametrize("m", [1, 2, 3, 5, 8, 13, 16])
def test_token_counts(q4k, m):
    _check(q4k, 256, 512, m, 10 + m)


@pytest.mark.parametrize("m", [1, 4, 16])
def test_q8_input_bf16(q4k, m):
    _check(q4k, 384, 768, m, 30 + m, out="bf16", act="q8", kind="outlier")


@pytest.mark.parametrize("n,k,m,out", [(4096, 4096, 1, "bf16"), (11008, 4096, 4, "bf16"), (4096, 11008, 16, "f32")])
def test_decode_sizes(q4k, n, k, m, out):
    """7B projection shapes (every output checked; 11008 rows give the
    persistent CTAs several row groups each)."""
    _check(q4k, n, k, m, 50 + m, out=out, kind="silu_mul" if k == 11008 else "normal")


@pytest.mark.parametrize("n,k,m,out", [(4096, 11008, 1, "bf16"), (128, 256, 2, "f32"), (640, 2304, 3, "f32"),
                                       (640, 2304, 6, "f32"), (512, 11008, 12, "bf16"), (11008, 4096, 8, "bf16")])
def test_streamed_shapes(q4k, n, k, m, out):
    """Shapes of the streamed small-M kernel: 43 super-blocks (a short last
    stage of 3), one super-block, 9 super-blocks over 40 row groups; the
    tensor-core form with 6 and 8 tokens, and 12 tokens of k = 11008 (two
    passes of 8 tokens)."""
    _check(q4k, n, k, m, 55 + m, out=out, kind="silu_mul" if k == 11008 else "normal")


@pytest.mark.parametrize("m", [1, 3, 4])
def test_in_kernel_quantization_bits(q4k, m):
    n, k = 512, 2816
    blocks = inputs.q6k_blocks(n, k, 70 + m)
    x = inputs.activations(m, k, 70 + m, "outlier")
    packed = q4k.q6k_pack_weights(to_dev(blocks), n, k)
    xd = to_dev(x)
    a = q4k.q6k_gemm(packed, n, k, xd)
    q, da, ss = q4k.q8_quantize_rows(xd)
    b = q4k.q6k_gemm(packed, n, k, q, da=da, ssum=ss)
    c = q4k.q6k_gemm(packed, n, k, xd)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("m,n,k,out,act", [(17, 128, 256, "f32", "f32"), (64, 256, 512, "f32", "q8"),
                                            (200, 384, 768, "bf16", "f32"), (300, 256, 2816, "f32", "q8")])
def test_prefill_sizes_tensor_core_path(q4k, m, n, k, out, act):
    """m > 16: the tcgen05 GEMM with two fp16 weight planes (every output,
    ragged token tiles, the k-split of the last wave)."""
    _check(q4k, n, k, m, 90 + m, out=out, act=act, kind="outlier")


def test_prefill_chunk_integers_exact(q4k):
    """Every per-chunk accumulator of the tensor-core path equals the oracle's
    exact integer sum_s sc_s * sum (q - 32) * qa: the split of sc into its high
    and low bits and the fp32 accumulator lose nothing."""
    m, n, k = 64, 256, 512
    blocks = inputs.q6k_blocks(n, k, 5)
    x = inputs.activations(m, k, 5, "outlier")
    packed = q4k.q6k_pack_weights(to_dev(blocks), n, k)
    ws = torch.empty(q4k.q4k_act_workspace_bytes(m, k), dtype=torch.uint8, device=DEV)
    y = q4k.q6k_gemm(packed, n, k, to_dev(x), workspace=ws)   # leaves the fp16 operand in ws
    y2, acc = q4k.q6k_gemm_debug_chunk_acc(packed, n, k, ws, m)
    torch.cuda.synchronize()
    f = oq6.decode(blocks)
    qa, _, _ = oq8.quantize_rows(x)
    ints = oq6.chunk_ints(f, qa)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ints)
    assert torch.equal(y, y2)


def test_prefill_full_size_sampled(q4k):
    """2048 tokens through a 4096 x 11008 Q6_K matrix (a 7B down projection):
    sampled rows against the oracle."""
    from tests.gpu_common import sample_rows

    m, n, k = 2048, 4096, 11008
    blocks = inputs.q6k_blocks(n, k, 8)
    x = inputs.activations(m, k, 8, "silu_mul")
    packed = q4k.q6k_pack_weights(to_dev(blocks), n, k)
    y = q4k.q6k_gemm(packed, n, k, to_dev(x), out_dtype="bf16")
    torch.cuda.synchronize()
    rows = sample_rows(m, 4, 8)
    want, scale = _oracle(blocks, x[rows])
    assert_close(y.float().cpu().double().numpy()[rows], want, scale, "bf16", "q6k full size")


def test_small_m_too_large_for_shared_memory_takes_tensor_path(q4k):
    """16 tokens x 14336 do not fit the small-M kernel's shared memory: the
    call takes the tensor-core path instead and stays correct."""
    _check(q4k, 256, 14336, 16, 3, out="f32", act="f32")


def test_prefill_extreme_scales_exact(q4k):
    """The worst cases of the tensor-core path's exactness argument: rows with
    sc = -128 and q = 0 (sc * (q - 32) = 4096), sc = 127 and q = 63, sc = -128
    and q = 63, against tokens whose codes are all +127 or alternate +-127, so
    that a chunk's partial sums reach 32 * 4096 * 127 = 16,646,144 < 2^24.
    Every per-chunk integer equals the oracle's, every output is in bound."""
    m, n, k = 64, 128, 256
    q = np.zeros((n, k), dtype=np.uint8)
    sc = np.zeros((n, k // 16), dtype=np.int8)
    q[0:32], sc[0:32] = 0, -128
    q[32:64], sc[32:64] = 63, 127
    q[64:96], sc[64:96] = 63, -128
    rng = np.random.default_rng(17)
    q[96:] = rng.integers(0, 64, (32, k))
    sc[96:] = rng.integers(-128, 128, (32, k // 16))
    d_bits = np.full((n, k // 256), 0x1400, dtype=np.uint16)   # f16 2^-10
    blocks = oq6.encode(q, sc, d_bits)
    x = np.ones((m, k), dtype=np.float32)
    x[32:] *= np.where(np.arange(k) % 2 == 0, 1.0, -1.0).astype(np.float32)   # codes +127 / alternating
    packed = q4k.q6k_pack_weights(to_dev(blocks), n, k)
    ws = torch.empty(q4k.q4k_act_workspace_bytes(m, k), dtype=torch.uint8, device=DEV)
    y = q4k.q6k_gemm(packed, n, k, to_dev(x), out_dtype="f32", workspace=ws)
    _, acc = q4k.q6k_gemm_debug_chunk_acc(packed, n, k, ws, m)
    torch.cuda.synchronize()
    f = oq6.decode(blocks)
    qa, _, _ = oq8.quantize_rows(x)
    ints = oq6.chunk_ints(f, qa)
    assert ints[0, 0, 0] == 32 * 4096 * 127
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ints)
    want, scale = _oracle(blocks, x)
    assert_close(y.float().cpu().double().numpy(), want, scale, "f32", "q6k extreme scales")


def test_long_k_takes_the_register_held_kernel(q4k):
    """k = 20480 with 8 tokens: beyond the streamed kernel's shared memory, the
    register-held Q6_K kernel takes it; every output checked."""
    _check(q4k, 128, 20480, 8, 140, out="f32", act="q8")


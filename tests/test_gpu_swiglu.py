"""Gate/up pair GEMM with the SiLU(gate)*up epilogue (q4k_gemm_swiglu),
compared with the oracle.

The q8 codes of h decide the down projection's input, so they are checked bit
for bit: the oracle forms h from the same fp32 g and u the GPU product writes
(the pair GEMM with f32 output; the epilogue reads the same accumulators), with
its own fp32 SiLU in the fixed operation order, and quantizes it with its own
q8 rule.  g and u themselves are checked against the oracle's exact GEMM with
the usual bound, and the down projection fed from the epilogue's operand is
checked end to end.
"""
import numpy as np
import pytest
import torch

from oracle import gemm as ogemm
from oracle import q4k_blocks, q8 as oq8, swiglu as osw
from quantized_prefill_gemm_gb300 import inputs
from tests.gpu_common import DEV, assert_close, oracle_rows, sample_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4k():
    from quantized_prefill_gemm_gb300 import q4k as mod

    mod.q4k_device_error_word(reset=True)
    yield mod
    assert mod.q4k_device_error_word() == 0


def _pair_rows(n):
    """Packed row of gate output o and of up output o (the pair layout)."""
    o = np.arange(n)
    g = 128 * (o // 64) + 64 * ((o % 64) // 32) + (o % 32)
    return g, g + 32


def _bf16_rn_bits(v):
    """fp32 -> bf16 bits, round to nearest even (finite inputs)."""
    b = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def _operand(ws, m, k):
    """Split an operand workspace (q4k_act_quantize layout) into its arrays."""
    kc = k // 32
    mp = (m + 127) // 128 * 128
    align = lambda v: (v + 1023) // 1024 * 1024
    off_da = align(m * k * 2)
    off_e = align(off_da + mp * kc * 4)
    xq = ws[: m * k * 2].view(np.float16).reshape(m, k)
    dat = ws[off_da: off_da + mp * kc * 4].view(np.float32).reshape(mp // 128, kc, 128)
    da = dat.transpose(0, 2, 1).reshape(mp, kc)
    e = ws[off_e: off_e + 4 * m * kc].view(np.uint16).reshape(2, m, kc)
    return xq, da, e


def _check_operand(ws, h, rows, m):
    """The operand of an m-token batch, for tokens `rows` (h holds those rows),
    equals the oracle's q8 quantization of h; padding tokens have d_a = 0."""
    n = h.shape[1]
    xq, da, e = _operand(ws, m, n)
    qa, da_bits, ssum = oq8.quantize_rows(h)
    assert np.array_equal(xq[rows].astype(np.float32), qa.astype(np.float32)), "qa"
    want_da = da_bits.view(np.float16).astype(np.float32)
    assert np.array_equal(da[rows], want_da), "d_a"
    assert not da[m:].any(), "padding tokens must have d_a = 0"
    E = (want_da.astype(np.float64) * ssum.astype(np.float64)).astype(np.float32)   # exact
    hi = _bf16_rn_bits(E)
    lo = _bf16_rn_bits(E - (hi.astype(np.uint32) << 16).view(np.float32))
    assert np.array_equal(e[0][rows], hi) and np.array_equal(e[1][rows], lo), "d_a*ssum split"
    return qa, da_bits, ssum


def _case(n, k, m, seed):
    gate = inputs.q4k_blocks(n, k, seed, 11)
    up = inputs.q4k_blocks(n, k, seed, 12)
    x = inputs.activations(m, k, seed, "normal")
    return gate, up, x


@pytest.mark.parametrize("n,k,m", [(256, 512, 200), (512, 1024, 64), (256, 256, 1), (768, 512, 130)])
def test_swiglu_operand_bits_and_down_projection(q4k, n, k, m):
    gate, up, x = _case(n, k, m, 100 + m)
    packed = q4k.q4k_pack_swiglu_weights(to_dev(gate), to_dev(up), n, k)
    xd = to_dev(x)
    ygu = q4k.q4k_gemm(packed, 2 * n, k, xd, out_dtype="f32").cpu().numpy()
    h_ws = q4k.q4k_gemm_swiglu(packed, n, k, xd)
    torch.cuda.synchronize()
    gr, ur = _pair_rows(n)
    g, u = ygu[:, gr], ygu[:, ur]
    # g and u: the usual GEMM bound against the oracle
    rows = np.arange(m)
    want, scale = oracle_rows(gate, x, rows)
    assert_close(g.astype(np.float64), want, scale, "f32", "gate")
    want, scale = oracle_rows(up, x, rows)
    assert_close(u.astype(np.float64), want, scale, "f32", "up")
    # the epilogue's q8 operand: bit for bit
    h = osw.silu_mul(g, u)
    qa, da_bits, ssum = _check_operand(h_ws.cpu().numpy(), h, rows, m)
    # down projection fed by it
    nd = 256
    down = inputs.q4k_blocks(nd, n, 100 + m, 13)
    pd = q4k.q4k_pack_weights(to_dev(down), nd, n)
    y = q4k.q4k_gemm_quantized(pd, nd, n, h_ws, m, "f32")
    torch.cuda.synchronize()
    fields = q4k_blocks.decode(down)
    want = ogemm.gemm_blockwise(fields, qa, da_bits, ssum)
    scale = ogemm.abs_scale(fields, qa, da_bits)
    assert_close(y.cpu().double().numpy(), want, scale, "f32", "down projection")


def test_swiglu_q8_input_matches_f32_input(q4k):
    """The activation given as the q8 SoA, or already in operand form, gives
    the same operand bits."""
    n, k, m = 256, 512, 70
    gate, up, x = _case(n, k, m, 7)
    packed = q4k.q4k_pack_swiglu_weights(to_dev(gate), to_dev(up), n, k)
    xd = to_dev(x)
    a = q4k.q4k_gemm_swiglu(packed, n, k, xd)
    q, da, ss = q4k.q8_quantize_rows(xd)
    b = q4k.q4k_gemm_swiglu(packed, n, k, q, da=da, ssum=ss)
    c = q4k.q4k_gemm_swiglu_quantized(packed, n, k, q4k.q4k_act_quantize(xd), m)
    torch.cuda.synchronize()
    for other in (b, c):
        for xa, xb in zip(_operand(a.cpu().numpy(), m, n), _operand(other.cpu().numpy(), m, n)):
            assert np.array_equal(np.ascontiguousarray(xa).view(np.uint8), np.ascontiguousarray(xb).view(np.uint8))


def test_pair_packing_is_the_interleaved_packing(q4k):
    """Packing gate and up as a pair equals packing the row-interleaved matrix."""
    n, k = 192, 512
    gate = inputs.q4k_blocks(n, k, 3, 11)
    up = inputs.q4k_blocks(n, k, 3, 12)
    both = np.empty((2 * n,) + gate.shape[1:], dtype=gate.dtype)
    gr, ur = _pair_rows(n)
    both[gr] = gate
    both[ur] = up
    nb = q4k.q4k_swiglu_packed_bytes(n, k)
    assert nb == q4k.q4k_packed_bytes(2 * n, k)
    pa = torch.zeros(nb, dtype=torch.uint8, device=DEV)
    pb = torch.zeros(nb, dtype=torch.uint8, device=DEV)
    q4k.q4k_pack_swiglu_weights(to_dev(gate), to_dev(up), n, k, packed=pa)
    q4k.q4k_pack_weights(to_dev(both), 2 * n, k, packed=pb)
    torch.cuda.synchronize()
    assert torch.equal(pa, pb)


def test_swiglu_ffn_size_sampled(q4k):
    """The 7B FFN at the benchmark's size (2048 tokens, 11008 x 4096 gate and
    up, 4096 x 11008 down): every token's q8 operand bit for bit, g, u and the
    down projection on sampled tokens."""
    n, k, m = 11008, 4096, 2048
    gate, up, x = _case(n, k, m, 21)
    packed = q4k.q4k_pack_swiglu_weights(to_dev(gate), to_dev(up), n, k)
    xd = to_dev(x)
    ygu = q4k.q4k_gemm(packed, 2 * n, k, xd, out_dtype="f32").cpu().numpy()
    h_ws = q4k.q4k_gemm_swiglu(packed, n, k, xd)
    down = inputs.q4k_blocks(4096, n, 21, 13)
    pd = q4k.q4k_pack_weights(to_dev(down), 4096, n)
    y = q4k.q4k_gemm_quantized(pd, 4096, n, h_ws, m, "bf16")
    torch.cuda.synchronize()
    gr, ur = _pair_rows(n)
    g, u = ygu[:, gr], ygu[:, ur]
    rows = np.arange(m)
    qa, da_bits, ssum = _check_operand(h_ws.cpu().numpy(), osw.silu_mul(g, u), rows, m)
    srows = sample_rows(m, 3, 21)
    for blocks, got, what in ((gate, g, "gate"), (up, u, "up")):
        want, scale = oracle_rows(blocks, x, srows)
        assert_close(got[srows].astype(np.float64), want, scale, "f32", what)
    fields = q4k_blocks.decode(down)
    want = ogemm.gemm_blockwise(fields, qa[srows], da_bits[srows], ssum[srows])
    scale = ogemm.abs_scale(fields, qa[srows], da_bits[srows])
    assert_close(y.float().cpu().double().numpy()[srows], want, scale, "bf16", "down projection")

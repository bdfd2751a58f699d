"""Gate/up pair GEMM with the SiLU(gate)*up epilogue (q4k_gemm_swiglu),
compared with the oracle.

Two checks, one per reading of what must match:

* kernel specification: the q8 codes of h decide the down projection's input,
  so they are checked bit for bit.  Here the oracle forms h from the same fp32
  g and u the GPU product writes (the pair GEMM with f32 output; the epilogue
  reads the same accumulators), with its own fp32 SiLU in the fixed operation
  order, and quantizes it with its own q8 rule.  g and u themselves are checked
  against the oracle's exact GEMM with the usual bound.
* the FFN block from x alone (test_swiglu_chain_from_x_alone and the
  full-size test): the oracle computes g and u blockwise from x, h with the
  plain definition SiLU(g)*u = g/(1 + e^-g)*u in fp64, its q8 quantization and
  the down product; nothing of it comes from the GPU.  The GPU's operand may
  differ from the oracle's only where the error the GEMM bound allows in g and
  u can move h across a q8 rounding boundary (chain_accept below), and the
  down output must agree within the GEMM bound plus the exact effect of those
  code steps.
"""
import numpy as np
import pytest
import torch

from oracle import gemm as ogemm
from oracle import q4k_blocks, q8 as oq8, swiglu as osw
from quantized_prefill_gemm_gb300 import inputs
from tests.gpu_common import BF16_U, DEV, assert_close, oracle_rows, sample_rows, to_dev

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


SILU_LIP = 1.0999   # max |d SiLU(g)/dg| over all g (1.0998 at g = 2.3994)
EVAL_REL = 1e-6     # GPU fp32 SiLU*u vs the fp64 definition (test_oracle_swiglu pins 5e-7)
U32 = 2.0 ** -24


def gemm_error_bound(fields, qa, da_bits, ssum):
    """Bound on |g_gpu - g| of the GPU product, from its arithmetic: the chunk
    integers are exact; the fold, the super-block sum and the k-split sum are
    at most 128 fp32 roundings, each within 2^-24 of S = sum|w*a|; the min term
    Z = sum_c (d_a*ssum)(dmin*m) runs on bf16 hi/lo splits (each factor within
    2^-16, so 3*2^-16 per product) accumulated in fp32 over 3*kc products
    (2^-23 each, truncation allowed), relative to S_min = sum_c |d_a*ssum*dmin*m|."""
    kc = qa.shape[1] // 32
    s = ogemm.abs_scale(fields, qa, da_bits)
    e = np.abs(oq8.f16_bits_to_f64(da_bits) * ssum.astype(np.float64))                 # [M][kc]
    dmin = np.repeat(q4k_blocks.f16_bits_to_f64(fields["dmin_bits"]), 8, axis=1)        # [N][kc]
    s_min = e @ (dmin * fields["m"].astype(np.float64)).T
    return 128 * U32 * s + (3 * 2.0 ** -16 + 3 * kc * 2.0 ** -23) * s_min


def chain_oracle(gate, up, down, x):
    """The FFN block from x alone (fp64 wherever the pages fix no precision).

    Returns (h, q8 of h, down output, S of the down product, |dh| bound) for
    every row of x.  |dh| bounds |h_gpu - h| element by element from the
    products' error bound (gemm_error_bound) through SiLU's Lipschitz
    constant, plus the GPU's fp32 evaluation error and the fp32 rounding of h."""
    qx, dx, sx = oq8.quantize_rows(x)
    fg, fu, fd = q4k_blocks.decode(gate), q4k_blocks.decode(up), q4k_blocks.decode(down)
    g = ogemm.gemm_blockwise(fg, qx, dx, sx)
    u = ogemm.gemm_blockwise(fu, qx, dx, sx)
    dg = gemm_error_bound(fg, qx, dx, sx)
    du = gemm_error_bound(fu, qx, dx, sx)
    h = osw.silu_mul_f64(g, u)
    silu = osw.silu_mul_f64(g, np.ones_like(u))
    dh = SILU_LIP * dg * (np.abs(u) + du) + np.abs(silu) * du + (EVAL_REL + 2 * U32) * (np.abs(h) + 1e-30)
    h32 = h.astype(np.float32)
    qa, da_bits, ssum = oq8.quantize_rows(h32)
    y = ogemm.gemm_blockwise(fd, qa, da_bits, ssum)
    s = ogemm.abs_scale(fd, qa, da_bits)
    return h32, (qa, da_bits, ssum), y, s, dh


def chain_accept(h32, q8_or, dh, qa_gpu, da_gpu):
    """Every difference between the GPU's operand and the oracle's q8 of h must
    be one the stated bounds allow.  Per 32-element block with oracle amax A
    and inverse inv = 127/A, an error dh_k in h moves the pre-rounding value
    v_k = h_k * inv by at most eta_k = inv (dh_k + |h_k| max_j dh_j / A) (the
    second term: amax, hence inv, moves too) plus fp32 rounding; the GPU code
    must be a correct rounding of some value within eta_k of v_k, and its d_a
    the f16 rounding of some amax within max_j dh_j of A."""
    qa, da_bits, _ = q8_or
    m, k = h32.shape
    hb = h32.astype(np.float64).reshape(m, k // 32, 32)
    amax = np.abs(hb).max(axis=2)
    dmax = dh.reshape(m, k // 32, 32).max(axis=2)
    inv = 127.0 / np.maximum(amax - dmax, 1e-30)
    v = hb * (127.0 / amax)[:, :, None]
    eta = inv[:, :, None] * (dh.reshape(m, k // 32, 32) + np.abs(hb) * (dmax / amax)[:, :, None]) + 4 * 127 * U32
    qg = qa_gpu.astype(np.float64).reshape(m, k // 32, 32)
    bad = np.abs(qg - v) > 0.5 + eta
    assert not bad.any(), f"{int(bad.sum())} GPU codes not explained by the bounds"
    d_or = da_bits.view(np.float16).astype(np.float64)
    d_lo = ((amax - dmax) / 127.0).astype(np.float32).astype(np.float16).astype(np.float64)
    d_hi = ((amax + dmax) / 127.0).astype(np.float32).astype(np.float16).astype(np.float64)
    da_g = da_gpu.astype(np.float64)
    assert np.all((da_g >= d_lo) & (da_g <= d_hi)), "d_a outside the rounding of the allowed amax"
    flips = int((qg.reshape(m, k) != qa).sum())
    return flips, int((da_g != d_or).sum())


def check_chain(down, x_rows, y_gpu, qa_gpu, da_gpu, chain, out, what):
    """y_gpu (the down output of those rows) against the oracle chain."""
    h32, q8_or, y_or, s_or, dh = chain
    flips, dflips = chain_accept(h32, q8_or, dh, qa_gpu, da_gpu)
    w = np.abs(q4k_blocks.dequantize(q4k_blocks.decode(down)))
    qa, da_bits, _ = q8_or
    a_or = oq8.dequantize_rows(qa, da_bits)
    m, k = qa.shape
    a_g = (qa_gpu.astype(np.float64).reshape(m, k // 32, 32) * da_gpu.astype(np.float64)[:, :, None]).reshape(m, k)
    step = np.abs(a_g - a_or) @ w.T          # exact effect bound of the allowed code / scale steps
    s_g = np.abs(a_g) @ w.T
    tol = 1e-4 * np.maximum(s_or, s_g) + step
    if out == "bf16":
        tol = tol * (1.0 + BF16_U) + BF16_U * np.abs(y_or)
    err = np.abs(y_gpu - y_or)
    assert np.all(err <= tol), f"{what}: {int((err > tol).sum())} outside; worst {float((err / tol).max()):.3g}"
    return flips, dflips


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


@pytest.mark.parametrize("n,k,m", [(512, 1024, 200), (256, 512, 1), (1024, 768, 130)])
def test_swiglu_chain_from_x_alone(q4k, n, k, m):
    """x -> gate/up -> SiLU(g)*u -> q8 -> down on the GPU (fused pair GEMM
    with the SiLU epilogue, then the down GEMM from its operand), against the
    oracle chain computed from x alone with the plain fp64 SiLU."""
    gate, up, x = _case(n, k, m, 300 + m)
    down = inputs.q4k_blocks(256, n, 300 + m, 13)
    packed = q4k.q4k_pack_swiglu_weights(to_dev(gate), to_dev(up), n, k)
    pd = q4k.q4k_pack_weights(to_dev(down), 256, n)
    h_ws = q4k.q4k_gemm_swiglu(packed, n, k, to_dev(x))
    y = q4k.q4k_gemm_quantized(pd, 256, n, h_ws, m, "f32")
    torch.cuda.synchronize()
    xq, da, _ = _operand(h_ws.cpu().numpy(), m, n)
    chain = chain_oracle(gate, up, down, x)
    flips, _ = check_chain(down, x, y.cpu().double().numpy(), xq[:m], da[:m], chain, "f32", f"chain {n}x{k} m={m}")
    assert flips <= max(4, m * n // 1000)   # rounding straddles are rare


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
    yb = y.float().cpu().double().numpy()[srows]
    assert_close(yb, want, scale, "bf16", "down projection")
    # the same rows through the oracle chain from x alone
    xq, da, _ = _operand(h_ws.cpu().numpy(), m, n)
    chain = chain_oracle(gate, up, down, x[srows])
    check_chain(down, x[srows], yb, xq[srows], da[srows], chain, "bf16", "FFN chain, sampled rows")

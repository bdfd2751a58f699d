"""q8 activation quantization on the GPU vs the oracle: bit-exact q8, d_a, ssum."""
import numpy as np
import pytest
import torch

from oracle import q8 as oq8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4k():
    from quantized_prefill_gemm_gb300 import q4k as mod

    return mod


def _check(q4k, x):
    from tests.gpu_common import to_dev

    q, da, ss = q4k.q8_quantize_rows(to_dev(x))
    torch.cuda.synchronize()
    wq, wda, wss = oq8.quantize_rows(x)
    assert np.array_equal(q.cpu().numpy(), wq)
    assert np.array_equal(da.cpu().numpy().view(np.uint16), wda)
    assert np.array_equal(ss.cpu().numpy(), wss)


@pytest.mark.parametrize("m,k,kind,seed", [
    (64, 512, "normal", 0), (512, 4096, "normal", 1), (2630, 4096, "outlier", 2),
    (2048, 4096, "normal", 3), (2048, 11008, "silu_mul", 3), (1, 256, "normal", 9), (17, 32, "normal", 9)])
def test_q8_bit_exact_on_config_inputs(q4k, m, k, kind, seed):
    from quantized_prefill_gemm_gb300 import inputs

    _check(q4k, inputs.activations(m, k, seed, kind))


def test_q8_edge_blocks(q4k):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 256)).astype(np.float32)
    x[0] = 0.0                                             # all-zero row
    x[1, :32] = np.float32(2.0 ** -121)                    # below the 2^-120 cutoff: zero block
    x[1, 32:64] = np.float32(2.0 ** -119)                  # just above it
    x[2] = rng.integers(-127, 128, 256).astype(np.float32)  # exact integers, amax 127 per block
    x[2, ::32] = 127.0
    x[3] = np.float32(0.5) * np.arange(256, dtype=np.float32) - 64.0   # many exact .5 ties
    x[4] *= 1e4                                             # large magnitudes
    x[5] *= 1e-6                                            # f16-subnormal scales
    _check(q4k, x)


def test_q8_edge_blocks_large_batch(q4k):
    """The same special rows in a batch large enough (19,200 blocks) for the
    one-thread-per-block kernel (small batches use 8 lanes per block)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((600, 1024)).astype(np.float32)
    x[0::6] = 0.0
    x[1::6, :32] = np.float32(2.0 ** -121)
    x[1::6, 32:64] = np.float32(2.0 ** -119)
    x[2::6] = rng.integers(-127, 128, (100, 1024)).astype(np.float32)
    x[2::6, ::32] = 127.0
    x[3::6] = np.float32(0.5) * (np.arange(1024, dtype=np.float32) % 256) - 64.0
    x[4::6] *= 1e4
    x[5::6] *= 1e-6
    _check(q4k, x)


def test_q8_strided_rows(q4k):
    from quantized_prefill_gemm_gb300 import inputs

    from tests.gpu_common import DEV

    x = inputs.activations(33, 512, 5)
    big = torch.zeros((33, 640), dtype=torch.float32, device=DEV)
    big[:, :512] = torch.from_numpy(x).to(DEV)
    q, da, ss = q4k.q8_quantize_rows(big[:, :512])
    wq, wda, wss = oq8.quantize_rows(x)
    assert np.array_equal(q.cpu().numpy(), wq)
    assert np.array_equal(da.cpu().numpy().view(np.uint16), wda)
    assert np.array_equal(ss.cpu().numpy(), wss)


@pytest.mark.parametrize("m,k,ld", [
    (200, 512, 512),      # 16 blocks a token: whole warps
    (130, 768, 768),      # 24 blocks: the second warp of a token holds 8
    (3, 11008, 11264),    # 344 blocks (21.5 warps), strided rows
    (1, 256, 256),        # one 8-block token, 127 padding tokens
])
def test_act_operand_layout(q4k, m, k, ld):
    """The GEMM operand form in the workspace: fp16 qa, fp32 d_a per 128-token
    tile (zero for the padding tokens), and d_a*ssum split into two bf16 planes
    (hi + lo)."""
    from quantized_prefill_gemm_gb300 import inputs

    from tests.gpu_common import DEV, to_dev

    kc = k // 32
    x = inputs.activations(m, k, 7, "outlier")
    big = torch.full((m, ld), float("nan"), dtype=torch.float32, device=DEV)
    big[:, :k] = to_dev(x)
    ws = q4k.q4k_act_quantize(big[:, :k]).cpu().numpy()
    wq, wda, wss = oq8.quantize_rows(x)
    da = wda.view(np.float16).astype(np.float32)
    align = lambda v: (v + 1023) // 1024 * 1024
    off_da = align(m * k * 2)
    mp = (m + 127) // 128 * 128
    off_e = align(off_da + mp * kc * 4)
    xq = ws[: m * k * 2].view(np.float16).reshape(m, k)
    assert np.array_equal(xq.astype(np.float32), wq.astype(np.float32))
    dat = ws[off_da: off_da + mp * kc * 4].view(np.float32).reshape(mp // 128, kc, 128)
    got_da = dat.transpose(0, 2, 1).reshape(mp, kc)
    assert np.array_equal(got_da[:m], da)
    assert not got_da[m:].any()
    e = ws[off_e: off_e + 4 * m * kc].view(np.uint16).reshape(2, m, kc)
    bf = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    want = da.astype(np.float64) * wss.astype(np.float64)
    got = bf(e[0]) + bf(e[1])
    assert np.all(np.abs(got - want) <= 2.0 ** -16 * np.abs(want))

"""q4k_gemm for decode-sized batches (1 <= m <= 16 tokens): the CUDA-core
small-M path, compared with the oracle.

Same bar as the GEMM: per element |y_gpu - y_oracle| <= 1e-4 * sum_k |w_k a_k|
(plus one bf16 rounding for bf16 output).  The shapes span one and several
128-row tiles, a super-block count that is not a multiple of the kernel's 16
shares (k = 11008 has 43), every token count class (1, 2, 3-4, 5-8, 9-16),
both activation forms, and q8 arrays the path cannot take directly (it then
uses the general path).
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
                                       (11008, 4096, 16, "f32")])
def test_decode_sizes(q4k, n, k, m, out):
    """The 7B projections at decode batch sizes, every output checked."""
    _check(q4k, n, k, m, "silu_mul" if k == 11008 else "normal", 60 + m, out=out)


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

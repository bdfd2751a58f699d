"""q4k_gemm_static_workspace: the fused GEMM with the library's fixed device
workspace, called through the C ABI and compared with q4k_gemm (which takes a
caller-supplied workspace) on the same inputs.

This file is collected last on purpose: it must pass both in a fresh process
and after every other test has used the library.
"""
import numpy as np
import pytest
import torch

from tests.gpu_common import DEV, assert_close, make_case, oracle_rows, to_dev

MAX_BYTES = 64 << 20


def test_static_workspace_size_query():
    from quantized_prefill_gemm_gb300 import q4k

    assert q4k.q4k_static_workspace_bytes() == MAX_BYTES


@pytest.fixture(scope="module")
def q4k():
    from quantized_prefill_gemm_gb300 import q4k as mod

    mod.q4k_device_error_word(reset=True)
    yield mod
    assert mod.q4k_device_error_word() == 0


def _case(q4k, n, k, m, kind, seed, act, out):
    blocks, x = make_case(n, k, m, kind, seed)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    xd = to_dev(x)
    extra = {}
    if act == "q8":
        xd, da, ss = q4k.q8_quantize_rows(xd)
        extra = dict(da=da, ssum=ss)
    ref = q4k.q4k_gemm(packed, n, k, xd, out_dtype=out, **extra)
    ydt = torch.float32 if out == "f32" else torch.bfloat16
    y = torch.full((m, n), float("nan"), dtype=ydt, device=DEV)
    q4k.q4k_gemm_static_workspace(packed, n, k, xd, y, **extra)
    return blocks, x, ref, y


@pytest.mark.gpu
@pytest.mark.parametrize("calls", [
    # n, k, m, kind, seed, act, out: two calls in a row, the second reusing the
    # array the first left filled
    [(256, 1024, 300, "normal", 11, "f32", "f32"), (384, 512, 130, "outlier", 12, "q8", "bf16")],
    # small-M paths: m <= 4 with fp32 input quantizes in the product kernel (no
    # workspace); 4 < m <= 16 with fp32 input stages the q8 rows in the array
    [(256, 512, 3, "normal", 14, "f32", "f32"), (384, 1024, 9, "normal", 15, "f32", "bf16")],
])
def test_two_calls_match_q4k_gemm(q4k, calls):
    """Same kernels as q4k_gemm on the same inputs: the output is identical bit
    for bit, and within the test bound of the oracle."""
    for n, k, m, kind, seed, act, out in calls:
        blocks, x, ref, y = _case(q4k, n, k, m, kind, seed, act, out)
        torch.cuda.synchronize()
        assert torch.equal(y, ref), f"static vs q4k_gemm {n}x{k} m={m}: not bit-identical"
        ys = y.float().cpu().double().numpy()
        assert np.isfinite(ys).all()
        want, scale = oracle_rows(blocks, x, np.arange(m))
        assert_close(ys, want, scale, out, f"static vs oracle {n}x{k} m={m}")


@pytest.mark.gpu
def test_rejects_problem_beyond_the_array(q4k):
    """m * k whose workspace exceeds 64 MiB returns Q4K_ERR_WORKSPACE before
    any launch (buffers are real and sized for the shape regardless)."""
    n, k, m = 128, 8192, 4096
    assert q4k.q4k_gemm_workspace_bytes(m, n, k) > MAX_BYTES
    blocks, _ = make_case(n, k, 1, "normal", 13)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    x = torch.zeros((m, k), dtype=torch.float32, device=DEV)
    y = torch.zeros((m, n), dtype=torch.float32, device=DEV)
    with pytest.raises(q4k.Q4KError) as ei:
        q4k.q4k_gemm_static_workspace(packed, n, k, x, y)
    assert ei.value.status == 4   # Q4K_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 0).all())

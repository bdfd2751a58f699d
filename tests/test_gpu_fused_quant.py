"""q4k_gemm_inkernel_quant (the GEMM kernel quantizes fp32 x itself): it writes
the same operand bits as the separate pass (q4k_act_quantize), and its
product equals the one computed from that pass's operand bit for bit (the
shapes are chosen so that both orders of the output tiles split the same
tiles along k, or none), and matches the oracle within the bound.

The cases span one and several token tiles, a ragged last tile (padding
tokens), slices of uneven width (k = 11008), the k-split tail, shapes whose
first wave leaves token tiles to the background warps, and workspaces that
start with garbage or with a previous call's counts.
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


def _operand_end(m, k):
    """Bytes of the workspace holding xq, d_a and E (the region both forms write)."""
    align = lambda v: (v + 1023) // 1024 * 1024
    kc, mp = k // 32, (m + 127) // 128 * 128
    off_da = align(m * k * 2)
    off_e = align(off_da + mp * kc * 4)
    return off_e + 2 * m * kc * 2


def _ws(q4k, m, k, fill):
    nb = q4k.q4k_act_workspace_bytes(m, k)
    if fill == "random":
        g = torch.Generator(device=DEV).manual_seed(m * 7 + k)
        return torch.randint(0, 256, (nb,), dtype=torch.uint8, device=DEV, generator=g)
    return torch.full((nb,), fill, dtype=torch.uint8, device=DEV)


CASES = [
    (200, 256, 1024, "f32"),     # 2 token tiles, k-split tail, every item at the start
    (300, 11008, 4096, "bf16"),  # 86 output tiles: the first wave reads 2 of 3 token tiles
    (130, 4096, 11008, "f32"),   # 344 blocks in 64 slices of 5 or 6
    (2048, 256, 4096, "f32"),    # 16 token tiles, 4-way k-split
    (2758, 4096, 4096, "bf16"),  # 22 token tiles, 58 padding tokens
    (64, 4096, 4096, "f32"),     # one token tile, half of it padding
]


@pytest.mark.parametrize("m,n,k,out", CASES)
def test_fused_operand_and_output_bits(q4k, m, n, k, out):
    from quantized_prefill_gemm_gb300 import inputs

    x = inputs.activations_torch(m, k, seed=11, kind="outlier", device=DEV)
    packed = q4k.q4k_pack_weights(inputs.q4k_blocks_torch(n, k, seed=12, device=DEV), n, k)
    ws_sep = _ws(q4k, m, k, 0)
    q4k.q4k_act_quantize(x, workspace=ws_sep)
    y_sep = q4k.q4k_gemm_quantized(packed, n, k, ws_sep, m, out_dtype=out)
    ws_fused = _ws(q4k, m, k, 0)
    y_fused = q4k.q4k_gemm_inkernel_quant(packed, n, k, x, out_dtype=out, workspace=ws_fused)
    torch.cuda.synchronize()
    end = _operand_end(m, k)
    assert torch.equal(ws_fused[:end], ws_sep[:end])
    assert torch.equal(y_fused.view(torch.int16 if out == "bf16" else torch.int32),
                       y_sep.view(torch.int16 if out == "bf16" else torch.int32))


@pytest.mark.parametrize("fill", [0xFF, "random"])
def test_fused_garbage_and_reused_workspace(q4k, fill):
    """Counts in the workspace that belong to no call, or to the previous call
    on the same workspace, are never taken for this call's."""
    from quantized_prefill_gemm_gb300 import inputs

    m, n, k = 904, 4096, 4096
    packed = q4k.q4k_pack_weights(inputs.q4k_blocks_torch(n, k, seed=21, device=DEV), n, k)
    ws = _ws(q4k, m, k, fill)
    for rep in range(3):   # a new x each time on the same workspace
        x = inputs.activations_torch(m, k, seed=30 + rep, device=DEV)
        y = q4k.q4k_gemm_inkernel_quant(packed, n, k, x, workspace=ws)
        ws_ref = q4k.q4k_act_quantize(x)
        y_ref = q4k.q4k_gemm_quantized(packed, n, k, ws_ref, m)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32)), rep


def test_fused_against_oracle(q4k):
    """The oracle, on a ragged shape with outliers (every element)."""
    m, n, k = 150, 384, 1024
    blocks, x = make_case(n, k, m, "outlier", seed=61)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    y = q4k.q4k_gemm_inkernel_quant(packed, n, k, to_dev(x))
    torch.cuda.synchronize()
    y_or, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(y.cpu().double().numpy(), y_or, scale, "f32")


def test_fused_empty_batch(q4k):
    from quantized_prefill_gemm_gb300 import inputs

    n, k = 256, 512
    packed = q4k.q4k_pack_weights(inputs.q4k_blocks_torch(n, k, seed=1, device=DEV), n, k)
    x = inputs.activations_torch(8, k, seed=2, device=DEV)
    y = q4k.q4k_gemm_inkernel_quant(packed, n, k, x[:0])   # a no-op
    torch.cuda.synchronize()
    assert y.shape == (0, n)


@pytest.mark.parametrize("name", ["qproj512", "qproj2630", "ffn2048"])
def test_fused_full_size_configs_sampled(q4k, name):
    """The configurations that take fp32 activations, at full size, through the
    in-kernel quantization: sampled token rows (tile edges and the ragged tail
    included) against the oracle, in each configuration's output type."""
    from tests.gpu_common import CONFIGS, sample_rows

    c = CONFIGS[name]
    m = c["m"]
    rows = sample_rows(m, 24, c["seed"])
    for i, (n, k, kind) in enumerate(c["mats"]):
        blocks, x = make_case(n, k, m, kind, c["seed"], tag=i)
        packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
        y = q4k.q4k_gemm_inkernel_quant(packed, n, k, to_dev(x), out_dtype=c["out"])
        torch.cuda.synchronize()
        want, scale = oracle_rows(blocks, x, rows)
        assert_close(y.float().cpu().double().numpy()[rows], want, scale, c["out"], f"{name}[{i}] {m}x{n}x{k}")


def test_fused_strided_activations(q4k):
    """x as the first k columns of wider rows (ldx > k): the same bits as the
    contiguous copy."""
    from quantized_prefill_gemm_gb300 import inputs

    m, n, k, ld = 300, 1024, 4096, 4160
    x = inputs.activations_torch(m, k, seed=71, kind="outlier", device=DEV)
    big = torch.full((m, ld), float("nan"), dtype=torch.float32, device=DEV)
    big[:, :k] = x
    packed = q4k.q4k_pack_weights(inputs.q4k_blocks_torch(n, k, seed=72, device=DEV), n, k)
    y_strided = q4k.q4k_gemm_inkernel_quant(packed, n, k, big[:, :k], out_dtype="bf16")
    y_dense = q4k.q4k_gemm_inkernel_quant(packed, n, k, x.contiguous(), out_dtype="bf16")
    torch.cuda.synchronize()
    assert torch.equal(y_strided.view(torch.int16), y_dense.view(torch.int16))

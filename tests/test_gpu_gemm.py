"""q4k_gemm on the GPU vs the oracle.

Bar: per element |y_gpu - y_oracle| <= 1e-4 * sum_k |w_k * a_k| for fp32 output
(plus one bf16 rounding, 2^-8 |y|, for bf16 output), and the per-chunk integer
dot products bit-exact (debug hook).  Small shapes are compared in full; the
full-size workloads on sampled token rows (every row is independent, so the
oracle computes exactly those rows), in the launch configuration the
benchmark uses.
"""
import numpy as np
import pytest
import torch

from oracle import gemm as ogemm
from oracle import q4k_blocks, q8 as oq8

from tests.gpu_common import CONFIGS, DEV, assert_close, make_case, oracle_rows, sample_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4k():
    from quantized_prefill_gemm_gb300 import q4k as mod

    mod.q4k_device_error_word(reset=True)
    yield mod
    assert mod.q4k_device_error_word() == 0


def _run(q4k, blocks, x, n, k, out, act="f32"):
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    if act == "q8":
        q, da, ss = q4k.q8_quantize_rows(to_dev(x))
        y = q4k.q4k_gemm(packed, n, k, q, out_dtype=out, da=da, ssum=ss)
    else:
        y = q4k.q4k_gemm(packed, n, k, to_dev(x), out_dtype=out)
    torch.cuda.synchronize()
    return y.float().cpu().double().numpy()


def test_tiny_config_full_and_exact_chunks(q4k):
    """Tiny workload (256 od x 512 k, 64 tokens, q8 path, fp32): every output,
    and every per-chunk accumulator equals sc * sum(q * qa) exactly."""
    c = CONFIGS["tiny"]
    n, k, kind = c["mats"][0]
    m = c["m"]
    blocks, x = make_case(n, k, m, kind, c["seed"])
    y = _run(q4k, blocks, x, n, k, "f32", act="q8")
    want, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(y, want, scale, "f32", "tiny")
    # exact integer chunk sums
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    ws = q4k.q4k_act_quantize(to_dev(x))
    y2, acc = q4k.q4k_gemm_debug_chunk_acc(packed, n, k, ws, m)
    torch.cuda.synchronize()
    fields = q4k_blocks.decode(blocks)
    qa, _, _ = oq8.quantize_rows(x)
    dots = ogemm.chunk_dots(fields, qa) * fields["sc"].astype(np.int64)[None, :, :]
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), dots)
    assert np.array_equal(acc.cpu().numpy(), dots.astype(np.float32))   # integral, no rounding
    assert np.array_equal(y2.cpu().double().numpy(), y)                 # same kernel, same numbers


@pytest.mark.parametrize("m,n,k,out", [
    (1, 128, 256, "f32"), (15, 256, 512, "f32"), (17, 128, 768, "bf16"), (70, 384, 512, "f32"),
    (129, 256, 1024, "bf16"), (300, 512, 2304, "f32")])
def test_ragged_shapes_full(q4k, m, n, k, out):
    blocks, x = make_case(n, k, m, "outlier", seed=m + n + k)
    y = _run(q4k, blocks, x, n, k, out)
    want, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(y, want, scale, out, f"{m}x{n}x{k}")


def test_exact_chunks_ragged(q4k):
    m, n, k = 131, 256, 768
    blocks, x = make_case(n, k, m, "normal", seed=77)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    ws = q4k.q4k_act_quantize(to_dev(x))
    _, acc = q4k.q4k_gemm_debug_chunk_acc(packed, n, k, ws, m)
    fields = q4k_blocks.decode(blocks)
    qa, _, _ = oq8.quantize_rows(x)
    dots = ogemm.chunk_dots(fields, qa) * fields["sc"].astype(np.int64)[None, :, :]
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), dots)


@pytest.mark.parametrize("name", ["qproj512", "qproj2630", "ffn2048", "stack_layer0"])
def test_full_size_configs_sampled(q4k, name):
    c = CONFIGS[name]
    m = c["m"]
    rows = sample_rows(m, 40, c["seed"])
    for i, (n, k, kind) in enumerate(c["mats"]):
        blocks, x = make_case(n, k, m, kind, c["seed"], tag=i)
        y = _run(q4k, blocks, x, n, k, c["out"], act=c["act"])
        want, scale = oracle_rows(blocks, x, rows)
        assert_close(y[rows], want, scale, c["out"], f"{name}[{i}] {m}x{n}x{k}")


def test_q8_path_matches_f32_path(q4k):
    m, n, k = 200, 256, 1024
    blocks, x = make_case(n, k, m, "outlier", seed=5)
    y1 = _run(q4k, blocks, x, n, k, "f32", act="f32")
    y2 = _run(q4k, blocks, x, n, k, "f32", act="q8")
    assert np.array_equal(y1, y2)


def test_degenerate_inputs(q4k):
    from quantized_prefill_gemm_gb300 import inputs

    m, n, k = 40, 128, 512
    blocks = inputs.q4k_blocks(n, k, 3)
    # X = 0 -> y = 0 exactly
    y = _run(q4k, blocks, np.zeros((m, k), np.float32), n, k, "f32")
    assert not y.any()
    # sc = m = 0 -> y = 0 exactly
    f = q4k_blocks.decode(blocks)
    f0 = dict(f, sc=np.zeros_like(f["sc"]), m=np.zeros_like(f["m"]))
    x = inputs.activations(m, k, 3)
    y = _run(q4k, q4k_blocks.encode(**f0), x, n, k, "f32")
    assert not y.any()
    # q = 0 -> the min term alone
    fq = dict(f, q=np.zeros_like(f["q"]))
    bq = q4k_blocks.encode(**fq)
    y = _run(q4k, bq, x, n, k, "f32")
    want, scale = oracle_rows(bq, x, np.arange(m))
    assert_close(y, want, scale, "f32", "q=0")
    # exact integer case: d = dmin = 1, integer x with block amax 127 -> integer y
    rng = np.random.default_rng(1)
    fi = dict(f, d_bits=np.full_like(f["d_bits"], 0x3C00), dmin_bits=np.full_like(f["dmin_bits"], 0x3C00))
    xi = rng.integers(-127, 128, (m, k)).astype(np.float32)
    xi[:, ::32] = 127.0
    bi = q4k_blocks.encode(**fi)
    y = _run(q4k, bi, xi, n, k, "f32")
    w_int = fi["q"].astype(np.int64) * np.repeat(fi["sc"].astype(np.int64), 32, axis=1) \
        - np.repeat(fi["m"].astype(np.int64), 32, axis=1)
    want = (xi.astype(np.int64) @ w_int.T).astype(np.float64)
    scale = np.abs(xi.astype(np.float64)) @ np.abs(w_int.T.astype(np.float64))
    assert_close(y, want, scale, "f32", "integer case")


def test_output_guard_regions_untouched(q4k):
    m, n, k = 70, 256, 512
    blocks, x = make_case(n, k, m, "normal", seed=11)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    canary = -12345.0
    ybig = torch.full((m + 3, n + 16), canary, dtype=torch.float32, device=DEV)
    y = ybig[:m, :n]
    q4k.q4k_gemm(packed, n, k, to_dev(x), out_dtype="f32", y=y)
    torch.cuda.synchronize()
    yb = ybig.cpu().numpy()
    assert np.all(yb[:, n:] == canary) and np.all(yb[m:, :] == canary)
    want, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(yb[:m, :n].astype(np.float64), want, scale, "f32", "strided y")


def test_repeat_calls_are_identical(q4k):
    m, n, k = 256, 512, 1024
    blocks, x = make_case(n, k, m, "normal", seed=12)
    y1 = _run(q4k, blocks, x, n, k, "bf16")
    y2 = _run(q4k, blocks, x, n, k, "bf16")
    assert np.array_equal(y1, y2)


def test_bounded_wait_selftest(q4k):
    assert q4k.q4k_selftest_wait_timeout(2_000_000) == q4k.Q4K_ERR_TIMEOUT   # 2 ms limit
    assert q4k.q4k_device_error_word() == 0                                   # reset by the self-test


def test_k_split_tail_and_workspace_reuse(q4k):
    """Tiles left over after the last full wave are split along k into parts of
    whole super-blocks; each part stores its partial tile in the workspace and
    a fixup kernel adds them in part order.  16 tiles with 8 super-blocks each
    split 4 ways (parts of at least two super-blocks) on a 152-SM part: every
    output against the oracle, three calls on one workspace giving the same
    bits."""
    m, n, k = 256, 1024, 2048
    blocks, x = make_case(n, k, m, "outlier", seed=91)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    ws = q4k.q4k_act_quantize(to_dev(x))
    ys = [q4k.q4k_gemm_quantized(packed, n, k, ws, m, "f32") for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
    want, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(ys[0].cpu().double().numpy(), want, scale, "f32", "k-split tail")


def test_k_split_four_parts_ragged_token_tile(q4k):
    """200 tokens x 11520 outputs: 2 x 90 = 180 tiles, a whole wave of 152 and
    28 tail tiles, each split along k into 4 parts of 4 super-blocks (only
    the first with the min term); the second token tile is ragged, so the
    fixup meets padding rows.  Sampled token rows of both tiles against the
    oracle, in both output types, and the bits repeat."""
    m, n, k = 200, 11520, 4096
    blocks, x = make_case(n, k, m, "outlier", seed=77)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    ws = q4k.q4k_act_quantize(to_dev(x))
    y32 = [q4k.q4k_gemm_quantized(packed, n, k, ws, m, "f32") for _ in range(2)]
    y16 = q4k.q4k_gemm_quantized(packed, n, k, ws, m, "bf16")
    torch.cuda.synchronize()
    assert torch.equal(y32[0], y32[1])
    rows = np.array([0, 77, 127, 128, 163, 199])
    want, scale = oracle_rows(blocks, x, rows)
    assert_close(y32[0].cpu().double().numpy()[rows], want, scale, "f32", "4-way split f32")
    assert_close(y16.float().cpu().double().numpy()[rows], want, scale, "bf16", "4-way split bf16")


def test_long_k_min_term_boxes_and_exact_chunks(q4k):
    """K = 14080 (440 chunks): 110 main stages of 128 k and 7 min-term stages of
    64 chunks each, the last holding 56 chunks and reading zeros past kc; 150
    tokens leave the token tile ragged.  Every output against the oracle, and
    every per-chunk integer exact."""
    m, n, k = 150, 256, 14080
    blocks, x = make_case(n, k, m, "outlier", seed=123)
    y = _run(q4k, blocks, x, n, k, "f32")
    want, scale = oracle_rows(blocks, x, np.arange(m))
    assert_close(y, want, scale, "f32", "long k")
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    ws = q4k.q4k_act_quantize(to_dev(x))
    _, acc = q4k.q4k_gemm_debug_chunk_acc(packed, n, k, ws, m)
    torch.cuda.synchronize()
    fields = q4k_blocks.decode(blocks)
    qa, _, _ = oq8.quantize_rows(x)
    dots = ogemm.chunk_dots(fields, qa) * fields["sc"].astype(np.int64)[None, :, :]
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), dots)

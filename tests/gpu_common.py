"""Shared helpers for the GPU parity tests (imported by tests marked gpu)."""
import numpy as np
import torch

from oracle import gemm as ogemm
from oracle import q4k_blocks, q8 as oq8
from quantized_prefill_gemm_gb300 import inputs

DEV = torch.device("cuda:0")

# The five workloads: (name, m, [(n, k, act kind)], out dtype, activation path)
CONFIGS = {
    "tiny": dict(m=64, mats=[(256, 512, "normal")], out="f32", seed=0, act="q8"),
    "qproj512": dict(m=512, mats=[(4096, 4096, "normal")], out="f32", seed=1, act="f32"),
    "qproj2630": dict(m=2630, mats=[(4096, 4096, "outlier")], out="bf16", seed=2, act="f32"),
    "ffn2048": dict(m=2048, mats=[(11008, 4096, "normal"), (11008, 4096, "normal"), (4096, 11008, "silu_mul")],
                    out="bf16", seed=3, act="f32"),
    "stack_layer0": dict(m=2048, mats=[(4096, 4096, "normal")] * 4 + [(11008, 4096, "normal")] * 2
                         + [(4096, 11008, "normal")], out="bf16", seed=4, act="f32"),
}


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


BF16_U = 2.0 ** -8   # unit roundoff of bf16 (8 significant bits): |RN(v) - v| <= 2^-8 |v|


def tolerance(y_or, scale, out):
    """Acceptance bound per element: 1e-4 * sum|w*a| for fp32 output.

    bf16 output is RN(y32) of an fp32 value y32 within 1e-4*S of the oracle,
    so it adds one bf16 rounding of y32: |RN(y32) - y32| <= 2^-8 |y32| <=
    2^-8 (|y_or| + 1e-4*S)."""
    tol = 1e-4 * scale
    if out == "bf16":
        tol = tol * (1.0 + BF16_U) + BF16_U * np.abs(y_or)
    return tol


def oracle_rows(blocks, x, rows):
    """Oracle result for a subset of token rows (rows are independent)."""
    fields = q4k_blocks.decode(blocks)
    qa, da_bits, ssum = oq8.quantize_rows(x[rows])
    y = ogemm.gemm_blockwise(fields, qa, da_bits, ssum)
    s = ogemm.abs_scale(fields, qa, da_bits)
    return y, s


def assert_close(y_gpu, y_or, scale, out, what=""):
    tol = tolerance(y_or, scale, out)
    err = np.abs(y_gpu - y_or)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / np.maximum(tol, 1e-300)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} outside bound; worst at {i}: "
                             f"gpu {y_gpu[i]!r} oracle {y_or[i]!r} tol {tol[i]!r}")
    return float((err / np.maximum(scale, 1e-300)).max())


def sample_rows(m, count, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(m, size=min(count, m), replace=False).tolist())
    rows |= {0, m - 1, min(m - 1, 127), min(m - 1, 128)}   # tile edges and the ragged tail
    return np.array(sorted(rows))


def make_case(n, k, m, kind, seed, tag=0):
    blocks = inputs.q4k_blocks(n, k, seed, tag)
    x = inputs.activations(m, k, seed, kind, tag)
    return blocks, x

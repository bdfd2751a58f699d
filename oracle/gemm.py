"""Oracle: the Q4_K x q8 GEMM (test infrastructure only).

Y[t, o] = sum_k W[o, k] · X[t, k], with W in Q4_K and X quantized into q8
blocks of 32.  Per 32-k chunk c of super-block sb the result is an integer dot
product followed by the two-term rank-1 rescale:

    y[t,o] = sum_c  da[t,c] · ( d[o,sb]·sc[o,c]·I[t,o,c]  −  dmin[o,sb]·m[o,c]·ssum[t,c] )
    I[t,o,c] = sum_{k in c} q[o,k] · qa[t,k]                      (exact integer)

Sources: "34 · r31 — q-major sda scale-read repack", §1 Background (the A side
per token: d and ssum; the correction term is ssum times the A-side scale,
combined with the B-side min term −dmin·m) and §2 Principle (the B side per
(chunk, od row): d·sc and −dmin·m); "22 · r17 — Wide warp remap", §1 Background
(the two-term "rank-1 fold" of r15).  The dense brute force below computes the
same sum as a plain fp64 matmul of dequantized operands and is the pin for the
blockwise form (the per-block identity sum_k w_k·a_k = da·(d·sc·Σq·qa −
dmin·m·ssum)).

Everything is float64 from exact inputs; integer dot products go through
float64 matmuls, exact because every partial sum is an integer below 2^53.
"""
from __future__ import annotations

import numpy as np

from . import q4k_blocks, q8

QK_K = 256
SUB = 32


def _check(fields, qa):
    n, k = fields["q"].shape
    m, k2 = qa.shape
    if k != k2 or k % QK_K:
        raise ValueError("K mismatch or not a multiple of 256")
    return m, n, k


def chunk_dots(fields: dict, qa: np.ndarray) -> np.ndarray:
    """I[t, o, c] = sum_{k in chunk c} q[o,k]·qa[t,k] as int64 [M][N][K/32]."""
    m, n, k = _check(fields, qa)
    q = fields["q"].astype(np.float64)
    a = qa.astype(np.float64)
    out = np.empty((m, n, k // SUB), dtype=np.int64)
    for c in range(k // SUB):
        sl = slice(c * SUB, (c + 1) * SUB)
        out[:, :, c] = np.rint(a[:, sl] @ q[:, sl].T).astype(np.int64)
    return out


def gemm_blockwise(fields: dict, qa: np.ndarray, da_bits: np.ndarray, ssum: np.ndarray) -> np.ndarray:
    """The two-term rescale, chunk by chunk, in the pages' order: y fp64 [M][N]."""
    m, n, k = _check(fields, qa)
    q = fields["q"].astype(np.float64)
    a = qa.astype(np.float64)
    da = q8.f16_bits_to_f64(da_bits)                      # [M][K/32]
    ss = ssum.astype(np.float64)                          # [M][K/32]
    d = q4k_blocks.f16_bits_to_f64(fields["d_bits"])      # [N][K/256]
    dmin = q4k_blocks.f16_bits_to_f64(fields["dmin_bits"])
    sc = fields["sc"].astype(np.float64)                  # [N][K/32]
    mn = fields["m"].astype(np.float64)
    y = np.zeros((m, n), dtype=np.float64)
    for c in range(k // SUB):
        sb = c // (QK_K // SUB)
        sl = slice(c * SUB, (c + 1) * SUB)
        i_c = a[:, sl] @ q[:, sl].T                       # exact integers
        main = (d[:, sb] * sc[:, c])[None, :] * i_c
        mins = ss[:, c][:, None] * (dmin[:, sb] * mn[:, c])[None, :]
        y += da[:, c][:, None] * (main - mins)
    return y


def gemm_dense(fields: dict, qa: np.ndarray, da_bits: np.ndarray) -> np.ndarray:
    """Brute force: dequantize both operands to fp64 and multiply."""
    w = q4k_blocks.dequantize(fields)
    a = q8.dequantize_rows(qa, da_bits)
    return a @ w.T


def abs_scale(fields: dict, qa: np.ndarray, da_bits: np.ndarray) -> np.ndarray:
    """S[t, o] = sum_k |w[o,k]·a[t,k]|, the per-element error scale."""
    w = np.abs(q4k_blocks.dequantize(fields))
    a = np.abs(q8.dequantize_rows(qa, da_bits))
    return a @ w.T


def gemm_from_x(blocks: np.ndarray, x: np.ndarray):
    """Convenience: quantize X, decode W, return (y, S, (qa, da_bits, ssum), fields)."""
    fields = q4k_blocks.decode(blocks)
    qa, da_bits, ssum = q8.quantize_rows(x)
    y = gemm_blockwise(fields, qa, da_bits, ssum)
    s = abs_scale(fields, qa, da_bits)
    return y, s, (qa, da_bits, ssum), fields

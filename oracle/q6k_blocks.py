"""Oracle: the Q6_K super-block format and its blockwise product (test
infrastructure only).

Source: the series' Q6_K line is named in "34 · r31 — q-major sda scale-read
repack", §5 Results (the post-hoc notes), as the format the campaign moved
on to after Q4_K; the pages give no layout or formula for it.  Reading: the
public GGUF Q6_K format, 256 weights per super-block, 210 bytes:
  bytes   0-127  ql[128]: the low 4 bits of the quants
  bytes 128-191  qh[64]:  the high 2 bits
  bytes 192-207  sc[16]:  one signed 8-bit scale per 16 weights
  bytes 208-209  d:       the super-block scale (f16, little endian)
with w = d * sc * (q - 32), q in 0..63.  Weights 128h .. 128h+127 (h = 0, 1)
use ql[64h ..], qh[32h ..] and sc[8h ..]; for l = 0..31:
  weight 128h + l      : q = (ql[64h+l]    & 15) | ((qh[32h+l] >> 0) & 3) << 4
  weight 128h + l + 32 : q = (ql[64h+l+32] & 15) | ((qh[32h+l] >> 2) & 3) << 4
  weight 128h + l + 64 : q = (ql[64h+l]    >> 4) | ((qh[32h+l] >> 4) & 3) << 4
  weight 128h + l + 96 : q = (ql[64h+l+32] >> 4) | ((qh[32h+l] >> 6) & 3) << 4
and weight 16j + i of the super-block (i < 16) has scale sc[j].
Parity unpinned for GGUF interop (no GGUF file here); every test goes through
this module's own encode/decode.

The product with q8 activations (32-element blocks with d_a and ssum, as for
Q4_K) follows the same per-block reading as the Q4_K path: per 32-k chunk c
(two 16-weight sub-blocks s), the exact integer
    I_c = sum_s sc_s * sum_{k in s} (q_k - 32) * qa_k,
then y = sum_c d_a[c] * d[sb(c)] * I_c.  There is no min term: the offset 32
is part of the integer.
"""
from __future__ import annotations

import numpy as np

from oracle import q8

QK_K = 256
SUB = 16
BLOCK_BYTES = 210


def decode(blocks: np.ndarray) -> dict:
    """Blocks [N][K/256][210] uint8 -> q uint8 [N][K] (0..63), sc int8 [N][K/16],
    d_bits uint16 [N][K/256]."""
    b = np.asarray(blocks, dtype=np.uint8)
    if b.ndim != 3 or b.shape[2] != BLOCK_BYTES:
        raise ValueError("blocks must be [N][K/256][210] uint8")
    n, nb, _ = b.shape
    ql = b[:, :, 0:128]
    qh = b[:, :, 128:192]
    sc = b[:, :, 192:208].view(np.int8)
    d_bits = b[:, :, 208].astype(np.uint16) | (b[:, :, 209].astype(np.uint16) << 8)
    q = np.zeros((n, nb, QK_K), dtype=np.uint8)
    for h in range(2):
        lo = ql[:, :, 64 * h: 64 * h + 64]
        hi = qh[:, :, 32 * h: 32 * h + 32]
        base = 128 * h
        q[:, :, base: base + 32] = (lo[:, :, 0:32] & 15) | (((hi >> 0) & 3) << 4)
        q[:, :, base + 32: base + 64] = (lo[:, :, 32:64] & 15) | (((hi >> 2) & 3) << 4)
        q[:, :, base + 64: base + 96] = (lo[:, :, 0:32] >> 4) | (((hi >> 4) & 3) << 4)
        q[:, :, base + 96: base + 128] = (lo[:, :, 32:64] >> 4) | (((hi >> 6) & 3) << 4)
    return {"q": q.reshape(n, nb * QK_K), "sc": np.ascontiguousarray(sc).reshape(n, nb * 16),
            "d_bits": np.ascontiguousarray(d_bits)}


def encode(q, sc, d_bits) -> np.ndarray:
    """Inverse of decode."""
    q = np.asarray(q, dtype=np.uint8)
    n, k = q.shape
    if k % QK_K or np.any(q > 63):
        raise ValueError("q must be [N][K] with K % 256 == 0 and values 0..63")
    nb = k // QK_K
    qb = q.reshape(n, nb, QK_K)
    out = np.zeros((n, nb, BLOCK_BYTES), dtype=np.uint8)
    for h in range(2):
        base = 128 * h
        w0, w1 = qb[:, :, base: base + 32], qb[:, :, base + 32: base + 64]
        w2, w3 = qb[:, :, base + 64: base + 96], qb[:, :, base + 96: base + 128]
        out[:, :, 64 * h: 64 * h + 32] = (w0 & 15) | ((w2 & 15) << 4)
        out[:, :, 64 * h + 32: 64 * h + 64] = (w1 & 15) | ((w3 & 15) << 4)
        out[:, :, 128 + 32 * h: 128 + 32 * h + 32] = (w0 >> 4) | ((w1 >> 4) << 2) | ((w2 >> 4) << 4) | ((w3 >> 4) << 6)
    out[:, :, 192:208] = np.asarray(sc, dtype=np.int8).reshape(n, nb, 16).view(np.uint8)
    d = np.asarray(d_bits, dtype=np.uint16).reshape(n, nb)
    out[:, :, 208] = (d & 0xFF).astype(np.uint8)
    out[:, :, 209] = (d >> 8).astype(np.uint8)
    return out


def dequantize(fields: dict) -> np.ndarray:
    """w = d * sc * (q - 32), exact in float64, [N][K]."""
    q = fields["q"].astype(np.float64)
    n, k = q.shape
    d = q8.f16_bits_to_f64(fields["d_bits"])                       # [N][K/256]
    sc = fields["sc"].astype(np.float64)                           # [N][K/16]
    return (q - 32.0) * np.repeat(sc, SUB, axis=1) * np.repeat(d, QK_K, axis=1)


def chunk_ints(fields: dict, qa: np.ndarray) -> np.ndarray:
    """I[t][o][c] = sum_s sc_s * sum_{k in s} (q - 32) * qa, exact (int64)."""
    v = fields["q"].astype(np.int64) - 32                          # [N][K]
    n, k = v.shape
    a = np.asarray(qa, dtype=np.int64)                             # [M][K]
    m = a.shape[0]
    sub = np.einsum("nsi,msi->mns", v.reshape(n, k // SUB, SUB), a.reshape(m, k // SUB, SUB))   # [M][N][K/16]
    sub = sub * fields["sc"].astype(np.int64)[None, :, :]
    return sub.reshape(m, n, k // 32, 2).sum(axis=3)               # [M][N][K/32]


def gemm_blockwise(fields: dict, qa: np.ndarray, da_bits: np.ndarray) -> np.ndarray:
    """y[t][o] = sum_c d_a[t,c] * d[o, sb(c)] * I[t][o][c], in float64."""
    ints = chunk_ints(fields, qa).astype(np.float64)               # [M][N][K/32]
    da = q8.f16_bits_to_f64(da_bits)                                # [M][K/32]
    d = np.repeat(q8.f16_bits_to_f64(fields["d_bits"]), 8, axis=1)  # [N][K/32]
    return np.einsum("mnc,mc,nc->mn", ints, da, d)


def abs_scale(fields: dict, qa: np.ndarray, da_bits: np.ndarray) -> np.ndarray:
    """S[t][o] = sum_k |w[o,k] * a[t,k]|, the per-element error scale."""
    w = np.abs(dequantize(fields))
    a = np.abs(q8.dequantize_rows(qa, da_bits))
    return a @ w.T

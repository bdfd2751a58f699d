"""Oracle: the Q4_K super-block format (test infrastructure only).

Source for the semantics: "34 · r31 — q-major sda scale-read repack", §2
Principle (the B side carries, per (chunk, od row), the pair d·sc and
−dmin·m), and the method statement: 256-weight super-blocks with f16 d and
dmin, eight 32-weight sub-blocks with a 6-bit scale sc and a 6-bit min m, and
4-bit quants q, so that w = d·sc·q − dmin·m.

The pages never print the byte layout.  Reading: the public GGUF Q4_K
arrangement, 144 bytes per super-block:
  bytes 0-1    d     (f16, little endian)
  bytes 2-3    dmin  (f16, little endian)
  bytes 4-15   s[0..11], the sixteen 6-bit fields:
                 sub-block j < 4:  sc = s[j] & 63,        m = s[j+4] & 63
                 sub-block j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4
                                   m  = (s[j+4] >> 4) | (s[j] >> 6) << 4
  bytes 16-143 qs[0..127]: for each pair of sub-blocks (2p, 2p+1), p = 0..3,
                 byte qs[32p + l] holds weight 64p + l in its low nibble and
                 weight 64p + 32 + l in its high nibble (l = 0..31).
Parity unpinned for GGUF interop (no GGUF file here); every test goes through
this module's own encode/decode, so results do not depend on the choice.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
SUB = 32
BLOCK_BYTES = 144


def decode(blocks: np.ndarray) -> dict:
    """Split blocks [N][K/256][144] uint8 into fields.

    Returns dict with q uint8 [N][K], sc uint8 [N][K/32], m uint8 [N][K/32],
    d_bits uint16 [N][K/256], dmin_bits uint16 [N][K/256].
    """
    b = np.asarray(blocks, dtype=np.uint8)
    if b.ndim != 3 or b.shape[2] != BLOCK_BYTES:
        raise ValueError("blocks must be [N][K/256][144] uint8")
    n, nb, _ = b.shape
    d_bits = b[:, :, 0].astype(np.uint16) | (b[:, :, 1].astype(np.uint16) << 8)
    dmin_bits = b[:, :, 2].astype(np.uint16) | (b[:, :, 3].astype(np.uint16) << 8)
    s = b[:, :, 4:16].astype(np.uint16)
    sc = np.zeros((n, nb, 8), dtype=np.uint8)
    m = np.zeros((n, nb, 8), dtype=np.uint8)
    for j in range(8):
        if j < 4:
            sc[:, :, j] = s[:, :, j] & 63
            m[:, :, j] = s[:, :, j + 4] & 63
        else:
            sc[:, :, j] = (s[:, :, j + 4] & 15) | ((s[:, :, j - 4] >> 6) << 4)
            m[:, :, j] = (s[:, :, j + 4] >> 4) | ((s[:, :, j] >> 6) << 4)
    qs = b[:, :, 16:144]
    q = np.zeros((n, nb, QK_K), dtype=np.uint8)
    for p in range(4):
        byte = qs[:, :, 32 * p: 32 * p + 32]
        q[:, :, 64 * p: 64 * p + 32] = byte & 15
        q[:, :, 64 * p + 32: 64 * p + 64] = byte >> 4
    return {
        "q": q.reshape(n, nb * QK_K),
        "sc": sc.reshape(n, nb * 8),
        "m": m.reshape(n, nb * 8),
        "d_bits": d_bits,
        "dmin_bits": dmin_bits,
    }


def encode(q, sc, m, d_bits, dmin_bits) -> np.ndarray:
    """Inverse of :func:`decode`: fields -> blocks [N][K/256][144] uint8."""
    q = np.asarray(q, dtype=np.uint8)
    n, k = q.shape
    nb = k // QK_K
    sc = np.asarray(sc, dtype=np.uint8).reshape(n, nb, 8)
    m = np.asarray(m, dtype=np.uint8).reshape(n, nb, 8)
    if q.max(initial=0) > 15 or sc.max(initial=0) > 63 or m.max(initial=0) > 63:
        raise ValueError("field out of range")
    d_bits = np.asarray(d_bits, dtype=np.uint16).reshape(n, nb)
    dmin_bits = np.asarray(dmin_bits, dtype=np.uint16).reshape(n, nb)
    out = np.zeros((n, nb, BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0] = d_bits & 0xFF
    out[:, :, 1] = d_bits >> 8
    out[:, :, 2] = dmin_bits & 0xFF
    out[:, :, 3] = dmin_bits >> 8
    s = np.zeros((n, nb, 12), dtype=np.uint16)
    for j in range(8):
        scj = sc[:, :, j].astype(np.uint16)
        mj = m[:, :, j].astype(np.uint16)
        if j < 4:
            s[:, :, j] |= scj
            s[:, :, j + 4] |= mj
        else:
            s[:, :, j + 4] |= (scj & 15) | ((mj & 15) << 4)
            s[:, :, j - 4] |= (scj >> 4) << 6
            s[:, :, j] |= (mj >> 4) << 6
    out[:, :, 4:16] = s.astype(np.uint8)
    qb = q.reshape(n, nb, QK_K)
    for p in range(4):
        lo = qb[:, :, 64 * p: 64 * p + 32]
        hi = qb[:, :, 64 * p + 32: 64 * p + 64]
        out[:, :, 16 + 32 * p: 16 + 32 * p + 32] = lo | (hi << 4)
    return out


def f16_bits_to_f64(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dequantize(fields: dict) -> np.ndarray:
    """w[o, k] = d·sc·q − dmin·m in float64 (exact: every factor is exact)."""
    q = fields["q"].astype(np.float64)
    n, k = q.shape
    d = np.repeat(f16_bits_to_f64(fields["d_bits"]), QK_K // SUB, axis=1)      # [N][K/32]
    dmin = np.repeat(f16_bits_to_f64(fields["dmin_bits"]), QK_K // SUB, axis=1)
    scale = d * fields["sc"].astype(np.float64)
    mins = dmin * fields["m"].astype(np.float64)
    w = q.reshape(n, k // SUB, SUB) * scale[:, :, None] - mins[:, :, None]
    return w.reshape(n, k)

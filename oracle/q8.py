"""Oracle: q8 activation quantization (test infrastructure only).

Source: "34 · r31 — q-major sda scale-read repack", §1 Background and §2
Principle: every q8 quantization block of the activations carries an f16
dequant scale d and an i16 ssum, the sum of the block's q8 values, and the two
feed the two-term rescale as a pair.

Readings where the page is silent (the rounding rule and op order are not
printed anywhere):
  * a block is 32 consecutive k of one token (the page's "32-token chunk" is
    read as a garble; its per-token layout indices and the 32-element q8 blocks
    of the method agree with this);
  * amax = max |x| over the block, in fp32;
  * d = RN32(amax / 127), inv = RN32(127 / amax);
  * qa = clamp(rint_half_even(RN32(x * inv)), -127, 127);
  * ssum = sum(qa) as int16; d_a = RN16(d) stored as f16 bits;
  * a block with amax < 2^-120 (where 127/amax would overflow fp32) is a zero
    block: qa = 0, ssum = 0, d_a = +0.
Inputs are finite; NaN / Inf are outside the domain.

All arithmetic is numpy float32 (IEEE, round-to-nearest-even, no FMA), so each
step is the single correctly rounded operation the reading names.
"""
from __future__ import annotations

import numpy as np

QK8 = 32
TINY_AMAX = np.float32(2.0 ** -120)


def quantize_rows(x: np.ndarray):
    """Quantize fp32 activations [M][K] into q8 blocks.

    Returns (qa int8 [M][K], da_bits uint16 [M][K/32] (f16 bit patterns),
    ssum int16 [M][K/32]).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % QK8:
        raise ValueError("x must be [M][K] with K a multiple of 32")
    m, k = x.shape
    xb = x.reshape(m, k // QK8, QK8)
    amax = np.max(np.abs(xb), axis=2)
    live = amax >= TINY_AMAX
    safe = np.where(live, amax, np.float32(1.0)).astype(np.float32)
    d = (safe / np.float32(127.0)).astype(np.float32)
    inv = (np.float32(127.0) / safe).astype(np.float32)
    v = (xb * inv[:, :, None]).astype(np.float32)
    q = np.clip(np.rint(v), -127.0, 127.0)
    q = np.where(live[:, :, None], q, 0.0).astype(np.int8)
    ssum = q.astype(np.int32).sum(axis=2).astype(np.int16)
    da = np.where(live, d, np.float32(0.0)).astype(np.float32).astype(np.float16)
    return q.reshape(m, k), da.view(np.uint16), ssum


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of f16 bit patterns as float64."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dequantize_rows(qa: np.ndarray, da_bits: np.ndarray) -> np.ndarray:
    """a = d_a * qa per block, exact in float64."""
    m, k = qa.shape
    da = f16_bits_to_f64(da_bits)
    return (qa.astype(np.float64).reshape(m, k // QK8, QK8) * da[:, :, None]).reshape(m, k)

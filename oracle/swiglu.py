"""Oracle: SiLU(gate)*up in fp32, the input of the down projection (test
infrastructure only).

Source: the pages measure "7B q4_K whole-prefill" ("34 · r31 — q-major sda
scale-read repack", Result), i.e. the linear layers of a LLaMA-7B model, whose
feed-forward block (SwiGLU: Shazeer, "GLU Variants Improve Transformer", 2020;
used by LLaMA, Touvron et al. 2023) feeds the down projection with
h = SiLU(g) * u, where g and u are the gate and up projections of the same
tokens and SiLU(g) = g / (1 + e^-g).  The pages print no formula or rounding
for it; this is the standard definition.

Reading (the pages are silent on precision): h is formed from the fp32 g and u
that the gate/up product writes, and the value that decides each q8 code must
be the same on both sides, so the evaluation order is fixed here, op by op,
in fp32 with round-to-nearest-even and no fused multiply-add.  With t = -g:

  t > 80:        SiLU = RN(g * 0) = -0          (true |SiLU| < 2e-33)
  t < -87:       SiLU = g                        (relative error < e^-87)
  otherwise:     s = RN(1 + E(t)),  SiLU = RN(g * R(s))
  h = RN(SiLU * u)

R(s) ~ 1/s is three Newton steps y <- RN(y * RN(2 - RN(s * y))) from the
seed y0 = the float whose bits are 0x7EF311C2 minus the bits of s (the
constant minimises the seed's largest relative error, 5.1%, over a binade);
within 2 ulp of 1/s for s in [1, 6e34], the range E gives here.  A division
would be the plainer choice; the reciprocal keeps the GPU's evaluation free of
branches, so that many elements are evaluated at once.

E(t) approximates e^t as follows (Cody and Waite's argument reduction,
"Software Manual for the Elementary Functions", 1980, with a Taylor
polynomial; constants are the mathematical values rounded to fp32):
  * t > 88: E = +inf (e^88 is 1.65e38; only g < -88 reaches it, where
    SiLU(g) = g / inf = -0 against a true |SiLU| < 1e-36);
  * t < -87: E = 0 (SiLU(g) = g, relative error below e^-87);
  * otherwise n = rint_even(RN(t * log2(e))), in [-126, 127];
    r = RN(RN(t - n*C1) - RN(n*C2)) with C1 = 355/512 (exact, so n*C1 is
    exact) and C2 = RN(ln 2 - C1);
    p = Horner form of sum_{j=0..7} r^j / j! (each step RN(RN(p*r) + c_j));
    E = RN(p * 2^n) with 2^n exact.
Accuracy (pinned by the tests against the fp64 exponential): within 2 ulp.

All arithmetic is numpy float32, each operation one IEEE operation.
"""
from __future__ import annotations

import numpy as np

F = np.float32
LOG2E = F(1.4426950408889634)
C1 = F(0.693359375)                                # 355 / 512
C2 = F(0.6931471805599453 - 0.693359375)           # ln 2 - C1
TAYLOR = [F(1.0 / f) for f in (5040.0, 720.0, 120.0, 24.0, 6.0, 2.0, 1.0, 1.0)]   # 1/7! .. 1/0!
T_INF = F(88.0)
T_ZERO = F(-87.0)
T_NEG = F(80.0)              # t = -g above this: SiLU is -0
RECIP_SEED = 0x7EF311C2


def exp_f32(t: np.ndarray) -> np.ndarray:
    """E(t) ~ e^t on fp32 input, in the fixed fp32 operation order above."""
    t = np.asarray(t, dtype=np.float32)
    mid = (t >= T_ZERO) & (t <= T_INF)
    tm = np.where(mid, t, F(0.0)).astype(np.float32)
    n = np.rint(tm * LOG2E).astype(np.float32)
    r = ((tm - n * C1).astype(np.float32) - (n * C2).astype(np.float32)).astype(np.float32)
    p = np.full_like(r, TAYLOR[0])
    for c in TAYLOR[1:]:
        p = ((p * r).astype(np.float32) + c).astype(np.float32)
    scale = np.ldexp(np.ones_like(n, dtype=np.float32), n.astype(np.int32)).astype(np.float32)   # exact 2^n
    e = (p * scale).astype(np.float32)
    e = np.where(t > T_INF, F(np.inf), e)
    e = np.where(t < T_ZERO, F(0.0), e)
    return e.astype(np.float32)


def recip_f32(s: np.ndarray) -> np.ndarray:
    """R(s) ~ 1/s for s in [1, 6e34]: bit-pattern seed, three Newton steps."""
    s = np.asarray(s, dtype=np.float32)
    bits = np.int64(RECIP_SEED) - s.view(np.uint32).astype(np.int64)
    y = bits.astype(np.uint32).view(np.float32)
    for _ in range(3):
        sy = (s * y).astype(np.float32)
        y = (y * (F(2.0) - sy).astype(np.float32)).astype(np.float32)
    return y


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = SiLU(g) * u in fp32, elementwise, in the order above."""
    g = np.asarray(g, dtype=np.float32)
    u = np.asarray(u, dtype=np.float32)
    t = (-g).astype(np.float32)
    e = exp_f32(np.minimum(t, T_NEG))
    s = (F(1.0) + e).astype(np.float32)
    silu = (g * recip_f32(s)).astype(np.float32)
    silu = np.where(t > T_NEG, (g * F(0.0)).astype(np.float32), silu)
    silu = np.where(t < T_ZERO, g, silu).astype(np.float32)
    return (silu * u).astype(np.float32)


def silu_mul_f64(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """The same function in float64 (the definition, for accuracy checks)."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * np.asarray(u, dtype=np.float64)

"""Seeded synthetic inputs for the Q4_K x q8 prefill GEMM.

This module only draws random numbers; it holds none of the GEMM's
arithmetic, so both the CUDA path and the CPU oracle can consume what it
makes without sharing any of the method.

Weights are random Q4_K super-blocks of 144 bytes per 256 weights (Q6_K:
210 bytes, see q6k_blocks).  Bytes 0-1
and 2-3 are the little-endian f16 words d and dmin, each drawn uniform on
[1e-3, 1e-2] and rounded to f16.  The other 140 bytes (sub-block scales and
mins, then the 4-bit quants) are uniform random bytes: in the Q4_K layout every
6-bit scale, 6-bit min and 4-bit quant is made of its own bits of these bytes,
so uniform bytes give uniform, independent fields (sc, m ~ U{0..63},
q ~ U{0..15}).

Activations are fp32 [tokens][k] matrices:
  * ``normal``   : N(0, 1)
  * ``outlier``  : N(0, 1) * (1 + 4 * B_k), B_k ~ Bernoulli(0.01) drawn once per
                   input channel k (about 1% outlier channels)
  * ``silu_mul`` : SiLU(G) * U with G, U ~ N(0, 1) independent (the shape of the
                   input a down projection sees after a SiLU-gated FFN)

Each buffer has its own stream, derived from (seed, tag), so a buffer does not
change when another one is added.  Host (numpy) and device (torch) generators
produce the same distributions, not the same numbers.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
BLOCK_BYTES = 144
D_LO, D_HI = 1e-3, 1e-2
OUTLIER_P = 0.01
OUTLIER_GAIN = 4.0

ACT_KINDS = ("normal", "outlier", "silu_mul")


def _rng(seed, tag) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tag)])


def q4k_blocks(n: int, k: int, seed: int, tag: int = 0) -> np.ndarray:
    """Random Q4_K weights, shape [n][k/256][144] uint8 (row-major, od rows)."""
    if k % QK_K:
        raise ValueError("k must be a multiple of 256")
    rng = _rng(seed, 1000 + tag)
    nb = k // QK_K
    blocks = rng.integers(0, 256, size=(n, nb, BLOCK_BYTES), dtype=np.uint8)
    scal = rng.uniform(D_LO, D_HI, size=(n, nb, 2)).astype(np.float16)
    blocks[:, :, 0:4] = scal.view(np.uint8).reshape(n, nb, 4)
    return blocks


Q6K_BLOCK_BYTES = 210
Q6K_D_LO, Q6K_D_HI = 1e-4, 1e-3


def q6k_blocks(n: int, k: int, seed: int, tag: int = 0) -> np.ndarray:
    """Random Q6_K weights, shape [n][k/256][210] uint8: uniform bytes for the
    quant bits and the int8 sub-block scales (so q ~ U{0..63}, sc ~ U{-128..127}),
    bytes 208-209 the f16 d ~ U[1e-4, 1e-3]."""
    if k % QK_K:
        raise ValueError("k must be a multiple of 256")
    rng = _rng(seed, 3000 + tag)
    nb = k // QK_K
    blocks = rng.integers(0, 256, size=(n, nb, Q6K_BLOCK_BYTES), dtype=np.uint8)
    d = rng.uniform(Q6K_D_LO, Q6K_D_HI, size=(n, nb, 1)).astype(np.float16)
    blocks[:, :, 208:210] = d.view(np.uint8).reshape(n, nb, 2)
    return blocks


def activations(m: int, k: int, seed: int, kind: str = "normal", tag: int = 0) -> np.ndarray:
    """Random fp32 activations, shape [m][k] row-major."""
    rng = _rng(seed, 2000 + tag)
    if kind == "normal":
        return rng.standard_normal((m, k), dtype=np.float32)
    if kind == "outlier":
        x = rng.standard_normal((m, k), dtype=np.float32)
        hot = _rng(seed, 3000 + tag).random(k) < OUTLIER_P
        gain = np.where(hot, np.float32(1.0 + OUTLIER_GAIN), np.float32(1.0)).astype(np.float32)
        return x * gain[None, :]
    if kind == "silu_mul":
        g = rng.standard_normal((m, k), dtype=np.float32)
        u = rng.standard_normal((m, k), dtype=np.float32)
        return (g / (np.float32(1.0) + np.exp(-g)) * u).astype(np.float32)
    raise ValueError(f"unknown activation kind {kind!r}")


# --------------------------------------------------------------------------
# Device-side generators (same distributions, drawn with torch on the GPU).
# Used for workloads too large to draw on the host in reasonable time.
# --------------------------------------------------------------------------

def _torch_gen(seed, tag, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(tag)) & ((1 << 63) - 1))
    return g


def q4k_blocks_torch(n: int, k: int, seed: int, tag: int = 0, device="cuda"):
    import torch

    if k % QK_K:
        raise ValueError("k must be a multiple of 256")
    g = _torch_gen(seed, 1000 + tag, device)
    nb = k // QK_K
    blocks = torch.randint(0, 256, (n, nb, BLOCK_BYTES), generator=g, device=device, dtype=torch.uint8)
    u = torch.empty((n, nb, 2), device=device, dtype=torch.float32).uniform_(D_LO, D_HI, generator=g)
    blocks[:, :, 0:4] = u.to(torch.float16).view(torch.uint8).reshape(n, nb, 4)
    return blocks


def q6k_blocks_torch(n: int, k: int, seed: int, tag: int = 0, device="cuda"):
    import torch

    if k % QK_K:
        raise ValueError("k must be a multiple of 256")
    g = _torch_gen(seed, 3000 + tag, device)
    nb = k // QK_K
    blocks = torch.randint(0, 256, (n, nb, Q6K_BLOCK_BYTES), generator=g, device=device, dtype=torch.uint8)
    u = torch.empty((n, nb, 1), device=device, dtype=torch.float32).uniform_(Q6K_D_LO, Q6K_D_HI, generator=g)
    blocks[:, :, 208:210] = u.to(torch.float16).view(torch.uint8).reshape(n, nb, 2)
    return blocks


def activations_torch(m: int, k: int, seed: int, kind: str = "normal", tag: int = 0, device="cuda"):
    import torch

    g = _torch_gen(seed, 2000 + tag, device)
    if kind == "normal":
        return torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
    if kind == "outlier":
        x = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
        hot = torch.rand((k,), generator=_torch_gen(seed, 3000 + tag, device), device=device) < OUTLIER_P
        return x * (1.0 + OUTLIER_GAIN * hot.to(torch.float32))[None, :]
    if kind == "silu_mul":
        gt = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
        u = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
        return gt / (1.0 + torch.exp(-gt)) * u
    raise ValueError(f"unknown activation kind {kind!r}")

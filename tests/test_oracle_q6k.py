"""Pins of the oracle's Q6_K format and blockwise product (CPU only).

The byte layout is written out here a second time, element by element from
the format table (not with the oracle's vectorised slicing), so that a wrong
shift, nibble or offset in the oracle's decoder fails; the product is pinned
to a dense fp64 brute force and to hand-evaluated values.
"""
import numpy as np

from oracle import q6k_blocks as q6
from oracle import q8 as oq8
from quantized_prefill_gemm_gb300 import inputs


def _encode_by_table(q, sc, d_bits):
    """One 210-byte block from fields, byte by byte from the layout table."""
    blk = bytearray(210)
    for h in range(2):
        for l in range(32):
            w = [q[128 * h + l + 32 * i] for i in range(4)]
            blk[64 * h + l] = (w[0] & 15) | ((w[2] & 15) << 4)
            blk[64 * h + 32 + l] = (w[1] & 15) | ((w[3] & 15) << 4)
            blk[128 + 32 * h + l] = (w[0] >> 4) | ((w[1] >> 4) << 2) | ((w[2] >> 4) << 4) | ((w[3] >> 4) << 6)
    for j in range(16):
        blk[192 + j] = sc[j] & 0xFF
    blk[208] = d_bits & 0xFF
    blk[209] = d_bits >> 8
    return np.frombuffer(bytes(blk), dtype=np.uint8).reshape(1, 1, 210)


def test_decode_matches_the_layout_table():
    rng = np.random.default_rng(11)
    for _ in range(20):
        q = rng.integers(0, 64, 256)
        sc = rng.integers(-128, 128, 16)
        d_bits = int(rng.integers(0, 0x7C00))
        f = q6.decode(_encode_by_table(q.tolist(), sc.tolist(), d_bits))
        assert np.array_equal(f["q"][0], q)
        assert np.array_equal(f["sc"][0], sc)
        assert int(f["d_bits"][0, 0]) == d_bits


def test_encode_decode_round_trip():
    b = inputs.q6k_blocks(16, 1024, 3)
    f = q6.decode(b)
    assert np.array_equal(q6.encode(f["q"], f["sc"], f["d_bits"]), b)


def test_worked_block_values():
    """q = i mod 64, sc_j = j - 8, d = 0.5 (f16 0x3800): w = 0.5 * sc * (q - 32)."""
    q = [i % 64 for i in range(256)]
    sc = [j - 8 for j in range(16)]
    f = q6.decode(_encode_by_table(q, sc, 0x3800))
    w = q6.dequantize(f)[0]
    assert w[0] == 0.5 * -8 * -32 == 128.0
    assert w[17] == 0.5 * -7 * (17 - 32) == 52.5
    assert w[255] == 0.5 * 7 * (63 - 32) == 108.5
    assert w[32] == 0.0 and w[96] == 0.0            # q = 32
    assert w[16 * 8 + 3] == 0.0                       # sc_8 = 0


def test_blockwise_equals_dense_brute_force():
    """sum_k w*a = sum_c d_a * d * sum_s sc_s * sum (q - 32) * qa, to fp64 rounding."""
    for seed, (n, k, m) in enumerate([(8, 256, 3), (16, 512, 5), (4, 2048, 2)]):
        f = q6.decode(inputs.q6k_blocks(n, k, seed))
        x = inputs.activations(m, k, seed, "outlier")
        qa, da, _ = oq8.quantize_rows(x)
        yb = q6.gemm_blockwise(f, qa, da)
        yd = oq8.dequantize_rows(qa, da) @ q6.dequantize(f).T
        s = q6.abs_scale(f, qa, da)
        assert np.all(np.abs(yb - yd) <= 1e-12 * s)


def test_chunk_integers_by_loops():
    f = q6.decode(inputs.q6k_blocks(2, 256, 7))
    qa = np.random.default_rng(7).integers(-127, 128, (2, 256)).astype(np.int8)
    ints = q6.chunk_ints(f, qa)
    for t in range(2):
        for o in range(2):
            for c in range(8):
                want = 0
                for k in range(32 * c, 32 * c + 32):
                    want += int(f["sc"][o, k // 16]) * (int(f["q"][o, k]) - 32) * int(qa[t, k])
                assert ints[t, o, c] == want


def test_degenerate_weights():
    x = inputs.activations(3, 256, 1)
    qa, da, _ = oq8.quantize_rows(x)
    q = np.full((2, 256), 32, dtype=np.uint8)                     # q - 32 = 0
    f = {"q": q, "sc": np.full((2, 16), 5, dtype=np.int8), "d_bits": np.full((2, 1), 0x3C00, dtype=np.uint16)}
    assert not q6.gemm_blockwise(f, qa, da).any()
    f = {"q": np.full((2, 256), 63, dtype=np.uint8), "sc": np.zeros((2, 16), dtype=np.int8),
         "d_bits": np.full((2, 1), 0x3C00, dtype=np.uint16)}
    assert not q6.gemm_blockwise(f, qa, da).any()

"""Pins for the CPU oracle (CPU only).

Each test checks the oracle against something other than itself: the IEEE f16
definition, hand-worked blocks (tests/golden/), a closed-form round-trip bound,
an exact integer GEMM, a dense fp64 brute force, and degenerate cases.  A
dropped term, a wrong sign, a transposed operand or a different rounding rule
anywhere in the oracle fails at least one of them.
"""
import os

import numpy as np
import pytest

from oracle import gemm, q4k_blocks, q8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- f16 -----

def _f16_by_definition(bits):
    """IEEE 754 binary16 value of each bit pattern, from sign/exponent/fraction."""
    bits = bits.astype(np.int64)
    s = np.where(bits >> 15, -1.0, 1.0)
    e = (bits >> 10) & 31
    f = (bits & 1023).astype(np.float64)
    sub = f * 2.0 ** -24
    nor = (1024.0 + f) * np.exp2(e.astype(np.float64) - 25.0)
    return s * np.where(e == 0, sub, nor), e == 31


def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    want, special = _f16_by_definition(bits)
    got = q8.f16_bits_to_f64(bits)
    assert np.array_equal(got[~special], want[~special])
    assert np.array_equal(q4k_blocks.f16_bits_to_f64(bits)[~special], want[~special])


def test_f16_encode_round_to_nearest_even():
    # every pair of adjacent positive finite f16 values: the fp32 midpoint
    # must round to the neighbour with the even fraction, points just off the
    # midpoint to the nearer neighbour
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)
    hi = lo + 1
    vlo, _ = _f16_by_definition(lo)
    vhi, _ = _f16_by_definition(hi)
    mid = ((vlo + vhi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (vlo + vhi) / 2)  # exact in fp32
    even = np.where(lo % 2 == 0, lo, hi)
    assert np.array_equal(mid.astype(np.float16).view(np.uint16), even)
    below = np.nextafter(mid, np.float32(0))
    above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(below.astype(np.float16).view(np.uint16), lo)
    assert np.array_equal(above.astype(np.float16).view(np.uint16), hi)


# ----------------------------------------------------------------- q8 -----

def _parse_pairs(field, dtype):
    out = np.zeros(32, dtype=dtype)
    for tok in field.split():
        i, v = tok.split(":")
        out[int(i)] = dtype(float(v))
    return out


def _load_q8_golden():
    rows = []
    with open(os.path.join(GOLDEN, "q8_worked_blocks.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, xs, qs, ssum, da = [p.strip() for p in line.split("|")]
            rows.append((name, _parse_pairs(xs, np.float32), _parse_pairs(qs, np.float64).astype(np.int8),
                         int(ssum), int(da, 16)))
    return rows


def test_q8_worked_blocks():
    rows = _load_q8_golden()
    x = np.stack([r[1] for r in rows])
    qa, da_bits, ssum = q8.quantize_rows(x)
    for i, (name, _, q_want, s_want, da_want) in enumerate(rows):
        assert np.array_equal(qa[i], q_want), name
        assert int(ssum[i, 0]) == s_want, name
        assert int(da_bits[i, 0]) == da_want, name


def test_q8_integer_blocks_are_exact():
    # integer x in [-127, 127] with block amax 127: d_a = 1 and qa = x
    rng = np.random.default_rng(7)
    x = rng.integers(-127, 128, size=(5, 256)).astype(np.float32)
    x[:, ::32] = 127.0
    qa, da_bits, ssum = q8.quantize_rows(x)
    assert np.array_equal(qa.astype(np.float32), x)
    assert np.all(da_bits == 0x3C00)
    assert np.array_equal(ssum, x.reshape(5, 8, 32).sum(axis=2).astype(np.int16))


def test_q8_round_trip_bound_and_invariants():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 1024)) * rng.uniform(1e-3, 50, size=(64, 1))).astype(np.float32)
    qa, da_bits, ssum = q8.quantize_rows(x)
    xb = x.reshape(64, 32, 32).astype(np.float64)
    q = qa.reshape(64, 32, 32).astype(np.int64)
    amax = np.abs(xb).max(axis=2)
    d = amax / 127.0
    da = q8.f16_bits_to_f64(da_bits)
    err = np.abs(xb - da[:, :, None] * q)
    bound = (0.5 * d + 2.0 ** -11 * amax) * (1 + 2.0 ** -20)
    assert np.all(err <= bound[:, :, None])
    assert np.abs(q).max() <= 127
    # the element of largest magnitude lands on +-127 with its sign
    idx = np.abs(xb).argmax(axis=2)
    top = np.take_along_axis(q, idx[:, :, None], axis=2)[:, :, 0]
    sgn = np.sign(np.take_along_axis(xb, idx[:, :, None], axis=2)[:, :, 0])
    assert np.array_equal(top, (127 * sgn).astype(np.int64))
    assert np.array_equal(ssum.astype(np.int64), q.sum(axis=2))
    # d_a is RN16 of amax/127 within f16 precision
    assert np.all(np.abs(da - d) <= 2.0 ** -11 * d + 2.0 ** -25)


def test_q8_zero_and_tiny_blocks():
    x = np.zeros((3, 64), dtype=np.float32)
    x[1, :32] = np.float32(2.0 ** -121)      # 127/amax would overflow: zero block
    x[2, :32] = np.float32(2.0 ** -119)      # still quantized normally
    x[2, 32:] = -3.0
    qa, da_bits, ssum = q8.quantize_rows(x)
    assert not qa[0].any() and not da_bits[0].any() and not ssum[0].any()
    assert not qa[1, :32].any() and da_bits[1, 0] == 0 and ssum[1, 0] == 0
    assert np.all(qa[2, :32] == 127) and ssum[2, 0] == 127 * 32
    assert np.all(qa[2, 32:] == -127) and ssum[2, 1] == -127 * 32


# ---------------------------------------------------------------- Q4_K ----

def _load_q4k_golden():
    g = {}
    with open(os.path.join(GOLDEN, "q4k_worked_block.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            g[key] = vals
    return g


def _golden_block():
    g = _load_q4k_golden()
    blk = np.zeros(144, dtype=np.uint8)
    d, dmin = int(g["d_bits"][0], 16), int(g["dmin_bits"][0], 16)
    blk[0], blk[1], blk[2], blk[3] = d & 255, d >> 8, dmin & 255, dmin >> 8
    blk[4:16] = [int(v, 16) for v in g["scales"]]
    for p in range(4):
        for l in range(32):
            blk[16 + 32 * p + l] = ((l + p) % 16) | (((15 - l - p) % 16) << 4)
    return blk.reshape(1, 1, 144), g


def test_q4k_worked_block():
    blk, g = _golden_block()
    f = q4k_blocks.decode(blk)
    assert list(f["sc"][0]) == [int(v) for v in g["sc"]]
    assert list(f["m"][0]) == [int(v) for v in g["m"]]
    assert f["d_bits"][0, 0] == 0x3C00 and f["dmin_bits"][0, 0] == 0x3800
    for tok in g["q"]:
        i, v = tok.split(":")
        assert f["q"][0, int(i)] == int(v)
    w = q4k_blocks.dequantize(f)
    for tok in g["w"]:
        i, v = tok.split(":")
        assert w[0, int(i)] == float(v)
    assert np.array_equal(q4k_blocks.encode(**f), blk)


def test_q4k_round_trip_random():
    rng = np.random.default_rng(3)
    n, k = 7, 768
    fields = {
        "q": rng.integers(0, 16, (n, k)).astype(np.uint8),
        "sc": rng.integers(0, 64, (n, k // 32)).astype(np.uint8),
        "m": rng.integers(0, 64, (n, k // 32)).astype(np.uint8),
        "d_bits": rng.integers(0, 0x7C00, (n, k // 256)).astype(np.uint16),
        "dmin_bits": rng.integers(0, 0x7C00, (n, k // 256)).astype(np.uint16),
    }
    blocks = q4k_blocks.encode(**fields)
    back = q4k_blocks.decode(blocks)
    for key in fields:
        assert np.array_equal(back[key], fields[key]), key
    raw = rng.integers(0, 256, (n, k // 256, 144)).astype(np.uint8)
    assert np.array_equal(q4k_blocks.encode(**q4k_blocks.decode(raw)), raw)


# ---------------------------------------------------------------- GEMM ----

def _random_case(m, n, k, seed):
    from quantized_prefill_gemm_gb300 import inputs

    blocks = inputs.q4k_blocks(n, k, seed)
    x = inputs.activations(m, k, seed)
    return blocks, x


def test_chunk_dots_brute_force():
    blocks, x = _random_case(3, 5, 256, 1)
    fields = q4k_blocks.decode(blocks)
    qa, _, _ = q8.quantize_rows(x)
    got = gemm.chunk_dots(fields, qa)
    for t in range(3):
        for o in range(5):
            for c in range(8):
                want = sum(int(fields["q"][o, k]) * int(qa[t, k]) for k in range(32 * c, 32 * c + 32))
                assert got[t, o, c] == want


@pytest.mark.parametrize("m,n,k", [(8, 16, 512), (5, 3, 768), (1, 32, 256)])
def test_blockwise_matches_dense_brute_force(m, n, k):
    blocks, x = _random_case(m, n, k, m * 100 + n)
    fields = q4k_blocks.decode(blocks)
    qa, da_bits, ssum = q8.quantize_rows(x)
    y = gemm.gemm_blockwise(fields, qa, da_bits, ssum)
    yd = gemm.gemm_dense(fields, qa, da_bits)
    s = gemm.abs_scale(fields, qa, da_bits)
    assert y.shape == (m, n)
    assert np.all(np.abs(y - yd) <= 1e-12 * s + 1e-300)


def test_exact_integer_gemm_special_case():
    # d = dmin = 1 and integer X with block amax 127 (so d_a = 1, qa = x):
    # y = sum_k (sc*q - m) * x exactly, an int64 matmul
    rng = np.random.default_rng(5)
    m, n, k = 6, 9, 512
    fields = {
        "q": rng.integers(0, 16, (n, k)).astype(np.uint8),
        "sc": rng.integers(0, 64, (n, k // 32)).astype(np.uint8),
        "m": rng.integers(0, 64, (n, k // 32)).astype(np.uint8),
        "d_bits": np.full((n, k // 256), 0x3C00, np.uint16),
        "dmin_bits": np.full((n, k // 256), 0x3C00, np.uint16),
    }
    x = rng.integers(-127, 128, (m, k)).astype(np.int64)
    x[:, ::32] = -127
    qa, da_bits, ssum = q8.quantize_rows(x.astype(np.float32))
    w_int = fields["q"].astype(np.int64) * np.repeat(fields["sc"].astype(np.int64), 32, axis=1) \
        - np.repeat(fields["m"].astype(np.int64), 32, axis=1)
    want = x @ w_int.T
    got = gemm.gemm_blockwise(fields, qa, da_bits, ssum)
    assert np.array_equal(got, want.astype(np.float64))


def test_degenerate_cases():
    blocks, x = _random_case(4, 8, 512, 9)
    fields = q4k_blocks.decode(blocks)
    # X = 0 -> y = 0 exactly
    qa0, da0, s0 = q8.quantize_rows(np.zeros_like(x))
    assert not gemm.gemm_blockwise(fields, qa0, da0, s0).any()
    qa, da_bits, ssum = q8.quantize_rows(x)
    # sc = m = 0 -> y = 0 exactly
    f0 = dict(fields, sc=np.zeros_like(fields["sc"]), m=np.zeros_like(fields["m"]))
    assert not gemm.gemm_blockwise(f0, qa, da_bits, ssum).any()
    # q = 0 -> only the min term: y = -sum_c da*ssum*dmin*m
    fq = dict(fields, q=np.zeros_like(fields["q"]))
    yq = gemm.gemm_blockwise(fq, qa, da_bits, ssum)
    dmin = np.repeat(q4k_blocks.f16_bits_to_f64(fields["dmin_bits"]), 8, axis=1)
    e = q8.f16_bits_to_f64(da_bits) * ssum.astype(np.float64)        # [M][C]
    want = -(e @ (dmin * fields["m"].astype(np.float64)).T)
    assert np.allclose(yq, want, rtol=1e-12, atol=0)
    # m = 0 (no min term) -> y = sum_c da*d*sc*I
    fm = dict(fields, m=np.zeros_like(fields["m"]))
    ym = gemm.gemm_blockwise(fm, qa, da_bits, ssum)
    assert np.allclose(ym, gemm.gemm_dense(fm, qa, da_bits), rtol=1e-12, atol=1e-300)


# ------------------------------------------------------- error scale S ----

def _load_abs_scale_golden():
    g = {}
    with open(os.path.join(GOLDEN, "abs_scale_worked.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            g[key] = vals
    return g


def _sparse(tokens, k, dtype):
    v = np.zeros(k, dtype=dtype)
    for tok in tokens:
        i, val = tok.split(":")
        v[int(i)] = float(val)
    return v


def test_abs_scale_worked_token():
    """S and y for one hand-worked token against the hand-worked block: the
    scale of every acceptance bound is pinned to a value worked out by hand."""
    blk, _ = _golden_block()
    g = _load_abs_scale_golden()
    fields = q4k_blocks.decode(blk)
    x = _sparse(g["x"], 256, np.float32)[None, :]
    qa, da_bits, ssum = q8.quantize_rows(x)
    assert np.array_equal(qa[0], _sparse(g["qa"], 256, np.int64).astype(np.int8))
    assert [int(v) for v in da_bits[0]] == [int(v, 16) for v in g["da_bits"]]
    assert [int(v) for v in ssum[0]] == [int(v) for v in g["ssum"]]
    w = q4k_blocks.dequantize(fields)
    for tok in g["w"]:
        i, v = tok.split(":")
        assert w[0, int(i)] == float(v)
    s = gemm.abs_scale(fields, qa, da_bits)
    assert s.shape == (1, 1) and s[0, 0] == float(g["S"][0])
    y = gemm.gemm_blockwise(fields, qa, da_bits, ssum)
    assert y[0, 0] == float(g["y"][0])
    assert gemm.gemm_dense(fields, qa, da_bits)[0, 0] == float(g["y"][0])


def test_abs_scale_explicit_loops():
    """S[t,o] = sum_k |w[o,k]| * |a[t,k]| by explicit loops over t, o, k, with
    w and a formed element by element from the fields (w = d*sc*q - dmin*m,
    a = d_a*qa): catches a dropped absolute value, a transposed operand or a
    wrong sign of the min term in the vectorised form."""
    rng = np.random.default_rng(17)
    m, n, k = 3, 4, 512
    blocks, x = _random_case(m, n, k, 17)
    x = x * rng.choice([-1.0, 1.0], size=x.shape).astype(np.float32)
    fields = q4k_blocks.decode(blocks)
    qa, da_bits, _ = q8.quantize_rows(x)
    d = q4k_blocks.f16_bits_to_f64(fields["d_bits"])
    dmin = q4k_blocks.f16_bits_to_f64(fields["dmin_bits"])
    da = q8.f16_bits_to_f64(da_bits)
    got = gemm.abs_scale(fields, qa, da_bits)
    for t in range(m):
        for o in range(n):
            acc = 0.0
            for kk in range(k):
                sb, c = kk // 256, kk // 32
                w = float(d[o, sb]) * int(fields["sc"][o, c]) * int(fields["q"][o, kk]) \
                    - float(dmin[o, sb]) * int(fields["m"][o, c])
                a = float(da[t, c]) * int(qa[t, kk])
                acc += abs(w * a)
            assert abs(got[t, o] - acc) <= 1e-12 * acc


def test_abs_scale_invariants():
    """S >= |y| (triangle inequality), with equality when every product has one
    sign: dmin*m = 0 and x >= 0 make every w*a >= 0, so S = y."""
    blocks, x = _random_case(5, 6, 768, 23)
    fields = q4k_blocks.decode(blocks)
    qa, da_bits, ssum = q8.quantize_rows(x)
    s = gemm.abs_scale(fields, qa, da_bits)
    y = gemm.gemm_blockwise(fields, qa, da_bits, ssum)
    assert np.all(s >= np.abs(y) * (1 - 1e-12))
    assert np.any(s > 1.01 * np.abs(y))   # random signs: strict somewhere
    f0 = dict(fields, m=np.zeros_like(fields["m"]))
    qp, dp, sp = q8.quantize_rows(np.abs(x))
    s0 = gemm.abs_scale(f0, qp, dp)
    y0 = gemm.gemm_blockwise(f0, qp, dp, sp)
    assert np.allclose(s0, y0, rtol=1e-12, atol=0)
    # S scales with the activations' d_a exactly: doubling x doubles every d_a
    qa2, da2, _ = q8.quantize_rows(2 * x)
    assert np.array_equal(qa2, qa)
    assert np.array_equal(gemm.abs_scale(fields, qa2, da2), 2 * s)

"""Pins of the oracle's fp32 SiLU(gate)*up against the mathematics (CPU only).

The fp32 function fixes the operation order that decides the q8 codes of the
down projection's input; these tests tie it to the exponential and to SiLU
themselves, so that a dropped reduction term, a wrong Taylor coefficient, a
sign error or a wrong threshold fails here rather than agreeing with a kernel
that shares the mistake.
"""
import math

import numpy as np

from oracle import swiglu as sw


def _ulp_err(got, want):
    got = np.asarray(got, dtype=np.float64)
    ulp = np.spacing(np.asarray(want, dtype=np.float32)).astype(np.float64)
    return np.abs(got - want) / ulp


def test_exp_within_1p5_ulp_of_exp_on_whole_range():
    t = np.linspace(-87.0, 88.0, 1_000_001, dtype=np.float32)
    err = _ulp_err(sw.exp_f32(t), np.exp(t.astype(np.float64)))
    assert err.max() <= 1.5, (err.max(), t[err.argmax()])


def test_exp_special_points():
    assert sw.exp_f32(np.float32(0.0)) == np.float32(1.0)
    # e^(n ln 2) is 2^n up to the rounding of ln 2 and of the result
    for n in (-120, -7, -1, 1, 9, 126):
        t = np.float32(n * math.log(2.0))
        want = math.exp(float(t))
        assert abs(float(sw.exp_f32(t)) - want) <= 2 * float(np.spacing(np.float32(want)))
    # the two cut-offs
    assert np.isinf(sw.exp_f32(np.float32(88.001)))
    assert np.isfinite(sw.exp_f32(np.float32(88.0)))
    assert sw.exp_f32(np.float32(-87.001)) == 0.0
    assert sw.exp_f32(np.float32(-87.0)) > 0.0
    # monotone on a fine grid around 0 and across reduction boundaries
    t = np.linspace(-3.0, 3.0, 200_001, dtype=np.float32)
    assert np.all(np.diff(sw.exp_f32(t).astype(np.float64)) >= 0.0)


def test_reciprocal_within_2_ulp():
    s = np.exp(np.linspace(0.0, np.log(6e34), 1_000_001)).astype(np.float32)
    err = _ulp_err(sw.recip_f32(s), 1.0 / s.astype(np.float64))
    assert err.max() <= 2.0, (err.max(), s[err.argmax()])
    # powers of two: the seed is already close, and the result is within 1 ulp
    p2 = np.float32(2.0) ** np.arange(0, 110, dtype=np.float32)
    assert _ulp_err(sw.recip_f32(p2), 1.0 / p2.astype(np.float64)).max() <= 1.0


def test_silu_mul_matches_definition():
    rng = np.random.default_rng(5)
    g = (rng.standard_normal(500_000) * 6.0).astype(np.float32)
    u = rng.standard_normal(500_000).astype(np.float32)
    got = sw.silu_mul(g, u).astype(np.float64)
    want = sw.silu_mul_f64(g, u)
    # a <= 1.5 ulp exponential, a <= 2 ulp reciprocal and three roundings
    assert np.all(np.abs(got - want) <= 5e-7 * np.abs(want) + 1e-32)


def test_silu_odd_part_identity():
    """SiLU(g) - SiLU(-g) = g for every g (SiLU(g) = g * sigmoid(g))."""
    g = np.linspace(-20.0, 20.0, 100_001, dtype=np.float32)
    one = np.ones_like(g)
    d = sw.silu_mul(g, one).astype(np.float64) - sw.silu_mul(-g, one).astype(np.float64)
    assert np.all(np.abs(d - g.astype(np.float64)) <= 5e-7 * np.abs(g.astype(np.float64)) + 1e-30)


def test_silu_limits():
    u = np.float32(3.0)
    assert sw.silu_mul(np.float32(0.0), u) == 0.0
    # large positive gate: SiLU(g) = g exactly
    assert sw.silu_mul(np.float32(95.5), u) == np.float32(95.5) * u
    # large negative gate: a signed zero
    z = sw.silu_mul(np.float32(-95.5), u)
    assert z == 0.0 and np.signbit(z)
    # just inside both cut-offs the general formula applies and is accurate
    for g in (-79.9, 86.9):
        got = float(sw.silu_mul(np.float32(g), np.float32(1.0)))
        want = float(np.float32(g)) / (1.0 + math.exp(-float(np.float32(g))))
        assert abs(got - want) <= 5e-7 * abs(want)
    # the value at g = 1: 1 / (1 + 1/e)
    assert abs(float(sw.silu_mul(np.float32(1.0), np.float32(1.0))) - 1.0 / (1.0 + math.exp(-1.0))) <= 2e-7


def test_silu_mul_f64_definition_values():
    """The fp64 form the FFN chain test takes as the definition: SiLU(0) = 0,
    SiLU(1) = 1/(1 + 1/e), SiLU(g) - SiLU(-g) = g, SiLU(g) -> g for large g and
    -> 0 for very negative g, and linearity in u."""
    one = np.ones(1)
    assert sw.silu_mul_f64(np.zeros(1), one)[0] == 0.0
    assert abs(sw.silu_mul_f64(one, one)[0] - 1.0 / (1.0 + math.exp(-1.0))) <= 1e-16
    g = np.linspace(-30.0, 30.0, 6001)
    u = np.ones_like(g)
    assert np.all(np.abs(sw.silu_mul_f64(g, u) - sw.silu_mul_f64(-g, u) - g) <= 1e-14 * (1.0 + np.abs(g)))
    assert sw.silu_mul_f64(np.array([60.0]), one)[0] == 60.0
    assert 0.0 > sw.silu_mul_f64(np.array([-60.0]), one)[0] > -1e-24
    assert sw.silu_mul_f64(np.array([2.0]), np.array([-3.0]))[0] == -3.0 * sw.silu_mul_f64(np.array([2.0]), one)[0]

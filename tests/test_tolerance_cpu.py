"""The bf16 term of the GPU acceptance bound, pinned on the CPU.

bf16 keeps 8 significant bits (7 stored), so one round-to-nearest-even step
moves a value by at most half an ulp, 2^-8 of the value's binade floor: the
relative error reaches 2^-8 (just above a power of two) and never exceeds it.
The GPU tests allow exactly one such rounding on top of the fp32 bound
(tests/gpu_common.py: tolerance); half of it (2^-9) would reject correct
roundings.
"""
import numpy as np
import torch

from tests.gpu_common import BF16_U, tolerance


def _rn_bf16(v):
    return torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()


def test_bf16_rounding_bound_is_2_pow_minus_8():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(1 << 20) * np.exp2(rng.integers(-20, 20, 1 << 20))).astype(np.float32)
    rel = np.abs(_rn_bf16(v) - v.astype(np.float64)) / np.abs(v.astype(np.float64))
    assert rel.max() <= BF16_U
    assert rel.max() > 0.99 * BF16_U          # the bound is reached
    # the worst case by construction: just below the midpoint above 1.0
    w = np.array([np.nextafter(np.float32(1.0 + 2.0 ** -8), np.float32(0.0))], dtype=np.float32)
    assert _rn_bf16(w)[0] == 1.0
    assert abs(1.0 - float(w[0])) > 2.0 ** -9 * float(w[0])


def test_tolerance_covers_one_rounding_of_any_value_within_the_fp32_bound():
    rng = np.random.default_rng(1)
    y_or = rng.standard_normal(1 << 16) * 10.0
    scale = np.abs(y_or) * rng.uniform(1.0, 100.0, y_or.shape)
    # the worst fp32 result the fp32 bound admits, then its bf16 rounding
    y32 = (y_or + np.sign(y_or) * 1e-4 * scale).astype(np.float32)
    got = _rn_bf16(y32)
    assert np.all(np.abs(got - y_or) <= tolerance(y_or, scale, "bf16"))
    assert np.array_equal(tolerance(y_or, scale, "f32"), 1e-4 * scale)

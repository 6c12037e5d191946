"""Pins for the oracle's RMS normalisation (queries and keys, per token, over d).

y = x / sqrt(mean(x^2) + eps) * w.  Pinned to: a hand-derived closed form, the
constant-vector closed form, mean(y^2) = 1 at eps = 0, scale invariance,
oddness, a 50-digit decimal brute force, the per-column role of the weight,
and a mutation test (sum instead of mean, dropped eps, weight applied per
row, missing square root) in which every broken restatement fails a pin.
"""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
from workloads import _rms_normalise, bf16_bits, bf16_to_f32, random_bf16


def pin_hand_closed_form(rms):
    # x = (3, 4): mean of squares 12.5, so y = (3, 4) / sqrt(12.5)
    y = rms(np.array([[3.0, 4.0]]), None, 0.0)
    np.testing.assert_allclose(y, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]], rtol=1e-15)


def pin_constant_vector(rms):
    c, eps, d = 0.37, 1e-3, 64
    y = rms(np.full((3, d), c), None, eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps), rtol=1e-14)


def pin_unit_mean_square(rms):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((50, 128)) * 7.0
    y = rms(x, None, 0.0)
    np.testing.assert_allclose((y ** 2).mean(-1), 1.0, rtol=0, atol=1e-14)


def pin_scale_invariance_and_oddness(rms):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((20, 64))
    y = rms(x, None, 0.0)
    np.testing.assert_allclose(rms(x * 123.0, None, 0.0), y, rtol=1e-13)
    np.testing.assert_allclose(rms(-x, None, 0.0), -y, rtol=1e-15)


def pin_decimal_bruteforce(rms):
    getcontext().prec = 50
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 6))
    w = rng.standard_normal(6)
    eps = 1e-2
    y = rms(x, w, eps)
    for r in range(4):
        ms = sum(Decimal(float(v)) ** 2 for v in x[r]) / 6
        inv = 1 / (ms + Decimal(eps)).sqrt()
        for c in range(6):
            want = Decimal(float(x[r, c])) * inv * Decimal(float(w[c]))
            assert abs(float(want) - y[r, c]) <= 1e-14 * max(1.0, abs(float(want)))


def pin_weight_per_column(rms):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 8))
    w = np.arange(1, 9, dtype=np.float64)
    np.testing.assert_allclose(rms(x, w, 1e-6), rms(x, None, 1e-6) * w[None, :], rtol=1e-15)


PINS = [pin_hand_closed_form, pin_constant_vector, pin_unit_mean_square,
        pin_scale_invariance_and_oddness, pin_decimal_bruteforce, pin_weight_per_column]


def real(x, w, eps):
    return oracle.rmsnorm(x, w, eps)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_rmsnorm_pin(pin):
    pin(real)


def test_bf16_inputs_widen_exactly():
    rng = np.random.default_rng(5)
    xb = random_bf16(rng, (7, 128), 2.0)
    np.testing.assert_array_equal(oracle.rmsnorm(xb, None, 1e-6),
                                  oracle.rmsnorm(bf16_to_f32(xb).astype(np.float64), None, 1e-6))


def test_generator_normalisation_agrees_with_oracle():
    # The input generator normalises in float32; it must agree with the oracle
    # to float32 rounding.
    rng = np.random.default_rng(6)
    x = rng.standard_normal((100, 128), dtype=np.float32)
    np.testing.assert_allclose(_rms_normalise(x).astype(np.float64),
                               oracle.rmsnorm(x.astype(np.float64), None, 1e-6), rtol=2e-6, atol=0)


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.rmsnorm(np.ones((2, 4)), None, -1.0)
    with pytest.raises(ValueError):
        oracle.rmsnorm(np.ones((2, 4)), np.ones(3), 0.0)


def _mut(kind):
    def f(x, w, eps):
        x = np.asarray(x, np.float64)
        ms = (x * x).sum(-1, keepdims=True) if kind == "sum" else (x * x).mean(-1, keepdims=True)
        e = 0.0 if kind == "no_eps" else eps
        inv = 1.0 / (ms + e) if kind == "no_sqrt" else 1.0 / np.sqrt(ms + e)
        y = x * inv
        if w is not None:
            y = y * (np.resize(w, (x.shape[0], 1)) if kind == "row_weight" else w[None, :])
        return y
    f.__name__ = kind
    return f


@pytest.mark.parametrize("kind", ["sum", "no_eps", "row_weight", "no_sqrt"])
def test_pins_catch_mutant(kind):
    failed = 0
    for pin in PINS:
        try:
            pin(_mut(kind))
        except AssertionError:
            failed += 1
    assert failed, kind


def test_unmutated_numpy_restatement_passes():
    for pin in PINS:
        pin(_mut("none"))

"""The polynomial exp2 the softmax evaluates on the FMA pipe, checked on the CPU.

The coefficients in ptx.cuh must be the ones the committed Remez script
derives, their relative error must stay within the stated bounds, and a
model of the device algorithm (each fp32 operation rounded as the GPU rounds
it: fma.sat, paired FMAs, the exponent added as an integer) must reproduce
2^x on [-125, 127] within the bound and clamp outside it.
"""
import importlib.util
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "diffusion_transformer_joint_causal_b300", "csrc")

# Relative-error bounds of the whole evaluation: the polynomial (1.73e-3,
# 7.5e-5) plus 1.3e-5 for the rounding of the clamped argument.
BOUND = {2: 1.75e-3, 3: 9.0e-5}


def _script():
    spec = importlib.util.spec_from_file_location("exp2_poly", os.path.join(CSRC, "exp2_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _header_coefficients():
    text = open(os.path.join(CSRC, "ptx.cuh")).read()
    out = {}
    for deg, n in ((2, 3), (3, 4)):
        out[deg] = np.array([float(re.search(rf"kExp2D{deg}C{i} = ([0-9.e+-]+)f", text).group(1))
                             for i in range(n)], dtype=np.float32)
    return out


@pytest.mark.parametrize("deg", [2, 3])
def test_header_coefficients_are_the_remez_ones(deg):
    derived = _script().fp32_coefficients(deg)
    assert np.array_equal(derived, _header_coefficients()[deg])


@pytest.mark.parametrize("deg,bound", [(2, 1.74e-3), (3, 7.6e-5)])
def test_minimax_error_is_levelled_and_bounded(deg, bound):
    mod = _script()
    c = mod.remez(deg)
    f = np.linspace(-0.5, 0.5, 200001)
    e = np.polynomial.polynomial.polyval(f, c) / np.exp2(f) - 1.0
    # equioscillation: deg + 2 extrema of alternating sign and equal size
    peaks = [e[0], e[-1]] + list(e[1:-1][(np.diff(np.sign(np.diff(e))) != 0)])
    assert len(peaks) >= deg + 2
    assert np.ptp(np.abs(peaks)) <= 1e-3 * np.max(np.abs(peaks))
    assert mod.max_rel_error_fp32(np.array(c, np.float32)) <= bound


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def _fma(a, b, c):
    # fp32 fused multiply-add: the exact product of two fp32 values fits in a
    # double, so one double sum rounded to fp32 models it (double rounding
    # could differ in rare ties; the bounds below leave room for that)
    return _f32(np.float64(a) * np.float64(b) + np.float64(c))


def exp2_model(x, deg):
    """Model of exp2_fma_pair for fp32 x."""
    coef = _header_coefficients()[deg]
    x = _f32(x)
    y = np.clip(_fma(x, np.float32(1 / 252), np.float32(125 / 252)), 0.0, 1.0).astype(np.float32)
    M = np.float32(12582912.0)
    t = _fma(y, np.float32(252), M - np.float32(125))
    nj = _fma(t, np.float32(-1), M - np.float32(125))
    f = _fma(y, np.float32(252), nj)
    p = np.full_like(f, coef[-1])
    for cm in coef[-2::-1]:
        p = _fma(p, f, cm)
    bits = (p.view(np.int32).astype(np.int64) + ((t.view(np.uint32).astype(np.int64) << 23)
                                                  & 0xFFFFFFFF)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("deg", [2, 3])
def test_model_matches_exp2_in_range(deg):
    rng = np.random.default_rng(1)
    x = np.concatenate([np.linspace(-125, 127, 500001), rng.uniform(-125, 127, 200000),
                        np.arange(-125, 128) + 0.5, np.arange(-125, 128) - 0.5,
                        np.arange(-125, 128).astype(float)])
    x = _f32(x)
    x = x[(x >= -125) & (x <= 127)]
    got = exp2_model(x, deg).astype(np.float64)
    rel = np.abs(got / np.exp2(x.astype(np.float64)) - 1.0)
    assert np.all(np.isfinite(got)) and float(rel.max()) <= BOUND[deg], float(rel.max())


@pytest.mark.parametrize("deg", [2, 3])
def test_model_clamps_outside_the_range(deg):
    lo = exp2_model(_f32([-126.0, -200.0, -1e30, -np.inf]), deg).astype(np.float64)
    hi = exp2_model(_f32([128.0, 300.0, 1e30, np.inf]), deg).astype(np.float64)
    assert np.all(np.abs(lo / 2.0 ** -125 - 1) <= BOUND[deg])
    assert np.all(np.abs(hi / 2.0 ** 127 - 1) <= BOUND[deg])
    # every result is a normal, finite float
    assert np.all(lo >= 2.0 ** -126) and np.all(np.isfinite(hi))


def test_model_notices_a_dropped_term():
    # the model is sensitive to the coefficients: dropping the last term
    # breaks the bound by orders of magnitude
    coef = _header_coefficients()[3]
    f = np.linspace(-0.5, 0.5, 1001)
    p = np.polynomial.polynomial.polyval(f, coef[:-1].astype(np.float64))
    assert np.max(np.abs(p / np.exp2(f) - 1)) > 100 * BOUND[3]

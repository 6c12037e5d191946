"""Pins for the FP64 oracle: facts fixed by the mathematics, not by the oracle.

The pages print no worked attention example, so the oracle is tied to:
  * a 50-digit decimal brute force of the definition on tiny, multi-head,
    Lq != Lk inputs (catches index, head-offset and operand mix-ups);
  * the two-key closed form o = v0 + (v1 - v0) * sigmoid(s1 - s0);
  * exact special cases: constant V, Lk = 1, scale = 0, one-hot selection
    with logits far beyond exp()'s overflow point;
  * invariants: rows of P sum to 1, key/value permutation invariance, query
    permutation equivariance, invariance under adding one vector to every key,
    outputs inside the convex hull of the value rows;
  * closed-form fixtures in tests/golden/closed_form.json.
Each pin is a function of an ``attn(q, k, v, scale)`` callable.  The last test
runs the pins against deliberately broken restatements of attention (dropped
scale, flipped exponent sign, swapped K/V, no max subtraction, wrong
normaliser, transposed head index) and checks that each one fails at least one
pin, so the pins are strong enough to catch a plausible mistake.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
from workloads import bf16_bits, bf16_to_f32, random_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def real_attn(q, k, v, scale):
    return oracle.attention(q, k, v, scale, n_threads=2)


def _as_f64(x):
    return bf16_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else np.asarray(x, np.float64)


# ----------------------------------------------------------------------------- pins

def pin_decimal_bruteforce(attn):
    """Definition evaluated with 50-digit decimals on B=2, H=2, Lq=5, Lk=7, d=3."""
    getcontext().prec = 50
    rng = np.random.default_rng(123)
    B, H, Lq, Lk, d = 2, 2, 5, 7, 3
    q = random_bf16(rng, (B, H, Lq, d), 1.5)
    k = random_bf16(rng, (B, H, Lk, d), 1.5)
    v = random_bf16(rng, (B, H, Lk, d))
    scale = float(np.float32(0.7))
    got = attn(q, k, v, scale)
    qf, kf, vf = (bf16_to_f32(x).astype(np.float64) for x in (q, k, v))
    D = lambda x: Decimal(float(x))  # exact: every float64 is a finite decimal
    for b in range(B):
        for h in range(H):
            for i in range(Lq):
                s = [D(scale) * sum(D(qf[b, h, i, c]) * D(kf[b, h, j, c]) for c in range(d))
                     for j in range(Lk)]
                m = max(s)
                p = [(x - m).exp() for x in s]
                l = sum(p)
                for c in range(d):
                    o = sum(p[j] * D(vf[b, h, j, c]) for j in range(Lk)) / l
                    assert abs(float(o) - got[b, h, i, c]) <= 1e-13, (b, h, i, c)


def pin_two_key_sigmoid(attn):
    """Lk = 2: o = v0 + (v1 - v0) * sigmoid(s1 - s0), s_j = scale * q.k_j."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, 6, 4))
    k = rng.standard_normal((1, 1, 2, 4))
    v = rng.standard_normal((1, 1, 2, 4))
    scale = 0.8
    got = attn(q, k, v, scale)
    for i in range(6):
        ds = scale * (float(q[0, 0, i] @ k[0, 0, 1]) - float(q[0, 0, i] @ k[0, 0, 0]))
        sig = 1.0 / (1.0 + math.exp(-ds))
        want = v[0, 0, 0] + (v[0, 0, 1] - v[0, 0, 0]) * sig
        np.testing.assert_allclose(got[0, 0, i], want, rtol=0, atol=1e-14)


def pin_constant_values(attn):
    """Every value row equal to c => every output row equals c."""
    rng = np.random.default_rng(1)
    q = random_bf16(rng, (1, 3, 9, 16))
    k = random_bf16(rng, (1, 3, 11, 16))
    c = np.float32(rng.standard_normal(16))
    v = np.broadcast_to(bf16_bits(c), (1, 3, 11, 16)).copy()
    got = attn(q, k, v, 0.25)
    np.testing.assert_allclose(got, np.broadcast_to(bf16_to_f32(bf16_bits(c)), got.shape),
                               rtol=1e-14, atol=0)


def pin_single_key(attn):
    """Lk = 1 => o_i = v_0 exactly, whatever the logits."""
    rng = np.random.default_rng(2)
    q = random_bf16(rng, (2, 2, 5, 8), 4.0)
    k = random_bf16(rng, (2, 2, 1, 8), 4.0)
    v = random_bf16(rng, (2, 2, 1, 8))
    got = attn(q, k, v, 1.0)
    want = np.broadcast_to(bf16_to_f32(v).astype(np.float64), got.shape)
    assert np.array_equal(got, want)


def pin_zero_scale_mean(attn):
    """scale = 0 => every probability is 1/Lk and o_i = mean_j v_j."""
    rng = np.random.default_rng(3)
    q = random_bf16(rng, (1, 2, 4, 8))
    k = random_bf16(rng, (1, 2, 13, 8))
    v = random_bf16(rng, (1, 2, 13, 8))
    got = attn(q, k, v, 0.0)
    want = bf16_to_f32(v).astype(np.float64).mean(axis=2, keepdims=True)
    np.testing.assert_allclose(got, np.broadcast_to(want, got.shape), rtol=0, atol=1e-15)


def pin_one_hot_selection(attn):
    """Q = alpha*e_pi(i), K = identity rows, alpha*scale = 1448 (beyond exp overflow).

    Query i then sees one logit 1448 and the rest 0, so o_i = v_pi(i) to within
    Lk*exp(-1448) -- and an implementation that skips the max subtraction
    overflows to inf/inf.
    """
    Lk = d = 8
    pi = np.array([3, 0, 7, 7, 1, 5, 2, 6, 4, 0])
    alpha = 4096.0  # exact in bf16
    qf = np.zeros((1, 1, len(pi), d), np.float32)
    qf[0, 0, np.arange(len(pi)), pi] = alpha
    kf = np.eye(Lk, d, dtype=np.float32)[None, None]
    rng = np.random.default_rng(4)
    v = random_bf16(rng, (1, 1, Lk, d))
    scale = float(np.float32(1 / math.sqrt(8)))
    got = attn(bf16_bits(qf), bf16_bits(kf), v, scale)
    want = bf16_to_f32(v).astype(np.float64)[0, 0, pi]
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got[0, 0], want, rtol=0, atol=1e-15)


def pin_rows_sum_to_one(attn_probs):
    rng = np.random.default_rng(5)
    q = random_bf16(rng, (1, 2, 17, 32), 2.0)
    k = random_bf16(rng, (1, 2, 29, 32), 2.0)
    v = random_bf16(rng, (1, 2, 29, 32))
    _, p = attn_probs(q, k, v, 0.3)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-14)


def pin_permutations(attn):
    """Permuting keys with values leaves O; permuting queries permutes O's rows."""
    rng = np.random.default_rng(6)
    q = random_bf16(rng, (2, 2, 12, 16), 1.5)
    k = random_bf16(rng, (2, 2, 19, 16), 1.5)
    v = random_bf16(rng, (2, 2, 19, 16))
    base = attn(q, k, v, 0.4)
    perm = rng.permutation(19)
    np.testing.assert_allclose(attn(q, k[:, :, perm], v[:, :, perm], 0.4), base,
                               rtol=0, atol=1e-13)
    qp = rng.permutation(12)
    np.testing.assert_allclose(attn(q[:, :, qp], k, v, 0.4), base[:, :, qp], rtol=0, atol=1e-15)


def pin_key_shift(attn):
    """Adding one vector u to every key shifts row i's logits by scale*q_i.u: O unchanged."""
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 2, 10, 8))
    k = rng.standard_normal((1, 2, 15, 8))
    v = rng.standard_normal((1, 2, 15, 8))
    u = rng.standard_normal(8) * 3.0
    np.testing.assert_allclose(attn(q, k + u, v, 0.5), attn(q, k, v, 0.5), rtol=0, atol=1e-12)


def pin_convex_hull(attn):
    rng = np.random.default_rng(9)
    q = random_bf16(rng, (1, 3, 20, 16), 3.0)
    k = random_bf16(rng, (1, 3, 31, 16), 3.0)
    v = random_bf16(rng, (1, 3, 31, 16))
    got = attn(q, k, v, 0.25)
    vf = bf16_to_f32(v).astype(np.float64)
    lo = vf.min(axis=2, keepdims=True) - 1e-15
    hi = vf.max(axis=2, keepdims=True) + 1e-15
    assert np.all(got >= lo) and np.all(got <= hi)


def pin_golden(attn):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = np.array(c["q"], np.float64)[None, None]
        k = np.array(c["k"], np.float64)[None, None]
        v = np.array(c["v"], np.float64)[None, None]
        got = attn(q, k, v, float(c["scale"]))[0, 0]
        want = np.array([[eval(x, {"__builtins__": {}}, {"e": math.e}) for x in row]  # noqa: S307
                         for row in c["o_closed_form"]])
        np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15, err_msg=c["name"])


PINS = [pin_decimal_bruteforce, pin_two_key_sigmoid, pin_constant_values, pin_single_key,
        pin_zero_scale_mean, pin_one_hot_selection, pin_permutations, pin_key_shift,
        pin_convex_hull, pin_golden]


# ----------------------------------------------------------------------------- tests

@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(real_attn)


def test_oracle_rows_sum_to_one():
    pin_rows_sum_to_one(lambda q, k, v, s: oracle.attention(q, k, v, s, return_probs=True))


def test_oracle_rows_subset_matches_full():
    rng = np.random.default_rng(10)
    q = random_bf16(rng, (2, 3, 40, 16))
    k = random_bf16(rng, (2, 3, 33, 16))
    v = random_bf16(rng, (2, 3, 33, 16))
    full = oracle.attention(q, k, v, 0.25, n_threads=3)
    bh = np.array([0, 5, 3, 3])
    rows = np.array([39, 0, 17, 18])
    sub = oracle.attention_rows(q, k, v, 0.25, bh, rows, n_threads=1)
    np.testing.assert_array_equal(sub, full.reshape(6, 40, 16)[bh, rows])


def test_oracle_rejects_bad_rows():
    q = np.zeros((1, 1, 4, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, 1.0, [0], [4])
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, 1.0, [1], [0])


# Broken restatements of attention: each must fail at least one pin.
def _mut_no_scale(q, k, v, scale):
    return _np_attn(q, k, v, 1.0)


def _mut_sign(q, k, v, scale):
    return _np_attn(q, k, v, scale, sign=-1.0)


def _mut_swap_kv(q, k, v, scale):
    return _np_attn(q, v, k, scale)


def _mut_no_max(q, k, v, scale):
    return _np_attn(q, k, v, scale, submax=False)


def _mut_norm_by_len(q, k, v, scale):
    return _np_attn(q, k, v, scale, norm="len")


def _mut_head_transpose(q, k, v, scale):
    kk = _as_f64(k)
    if kk.shape[0] > 1 or kk.shape[1] > 1:
        kk = kk[::-1, ::-1].copy()
    return _np_attn(q, kk, v, scale)


def _np_attn(q, k, v, scale, sign=1.0, submax=True, norm="sum"):
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    with np.errstate(over="ignore", invalid="ignore"):
        x = s - s.max(-1, keepdims=True) if submax else s
        p = np.exp(sign * x)
        l = p.sum(-1, keepdims=True) if norm == "sum" else s.shape[-1]
        return np.einsum("bhij,bhjd->bhid", p, v) / l


MUTANTS = [_mut_no_scale, _mut_sign, _mut_swap_kv, _mut_no_max, _mut_norm_by_len,
           _mut_head_transpose]


def test_numpy_restatement_passes_pins():
    # The unmutated numpy restatement must pass, or a mutant failing proves nothing.
    for pin in PINS:
        pin(_np_attn)


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_pins_catch_mutant(mutant):
    failed = []
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"

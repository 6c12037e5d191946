"""CPU checks of the tolerance the e4m3-probability path's GPU tests use.

The numerical model in fp8_model.py restates the kernel's arithmetic; these
tests check, against the FP64 oracle, that the model stays inside the
per-element bound and the aggregate relative-L2 bar of test_fp8_gpu.py on
diffuse and outlier-dominated rows, that it is exact where every probability
is exact in e4m3, and why the probability offset is 2^3 (at 2^4 most key
tiles would fail the optimistic pass on RMS-normalised logits).
"""
import math

import numpy as np

import fp8_model as M
import oracle
import workloads as W

REL_L2_FP8 = 4e-2


def _dequantised(rng, shape, gain_rows=None, gain=8.0, rms=False):
    x = W.bf16_to_f32(W.random_bf16(rng, shape))
    if rms:
        x = x / np.sqrt(np.mean(x.astype(np.float64) ** 2, axis=-1, keepdims=True)).astype(np.float32)
    if gain_rows is not None:
        x[..., gain_rows, :] *= gain
    codes, s = W.quantize_e4m3(x)
    return W.e4m3_to_f32(codes).astype(np.float64) * s


def _check(q, k, v, scale):
    """Model against the oracle for q [Lq, d], k, v [Lk, d]; returns (worst ratio, rel L2)."""
    ref = oracle.attention(q[None, None], k[None, None], v[None, None], scale)[0, 0]
    wabs = oracle.attention(q[None, None], k[None, None], np.abs(v)[None, None], scale)[0, 0]
    got = M.forward(scale * q @ k.T, v)
    err = np.abs(got - ref)
    return float(np.max(err / M.bound(wabs, ref))), float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def test_model_within_the_bound_on_diffuse_rows():
    rng = np.random.default_rng(5)
    q = _dequantised(rng, (200, 128), rms=True)
    k = _dequantised(rng, (3000, 128), rms=True)
    v = _dequantised(rng, (3000, 128))
    worst, rel = _check(q, k, v, float(np.float32(1 / math.sqrt(128))))
    assert worst <= 0.5 and rel <= REL_L2_FP8
    assert rel > 0.01          # the rounding of P is visible: the bar is not slack by orders


def test_model_within_the_bound_with_outlier_keys():
    rng = np.random.default_rng(6)
    Lk = 2000
    k_rows = rng.choice(Lk, 20, replace=False)
    q = _dequantised(rng, (200, 128))
    k = _dequantised(rng, (Lk, 128), gain_rows=k_rows)
    v = _dequantised(rng, (Lk, 128))
    worst, rel = _check(q, k, v, float(np.float32(1 / math.sqrt(128))))
    assert worst <= 1.0 and rel <= REL_L2_FP8


def test_model_exact_when_probabilities_are_exact():
    # one key per row 64 natural units above all others: p = 2^3 exactly and
    # the rest round to 0, so o is that key's value row (to the bf16 rounding)
    rng = np.random.default_rng(7)
    Lk, d = 300, 16
    s = np.zeros((50, Lk))
    pick = rng.integers(0, Lk, 50)
    s[np.arange(50), pick] = 64.0
    v = W.e4m3_to_f32(rng.integers(0, 0x7E, (Lk, d)).astype(np.uint8)).astype(np.float64)
    got = M.forward(s, v)
    # (keys of tiles before a row's key keep weights near 2^-92, as the
    # definition gives them e^-64)
    assert np.all(np.abs(got - v[pick]) <= 2.0 ** -8 * np.abs(v[pick]) + 1e-20)
    # equal logits: every p = 2^3, o = mean of the values
    got = M.forward(np.zeros((5, Lk)), v)
    assert np.allclose(got, v.mean(0), rtol=2.0 ** -8, atol=1e-12)


def test_offset_2_pow_3_keeps_the_optimistic_pass():
    # RMS-normalised logits of the 2048px workloads (s ~ N(0, 1)); the kernel
    # tests each thread's half-row sum (64 keys) against 448.  At an offset of
    # 2^5 that sum crosses 448 on about a tenth of the row tiles, at 2^3 never
    # (the rescale threshold keeps p <= 2^8 after a max pass in both).
    rng = np.random.default_rng(8)
    s = rng.standard_normal((256, 8192))
    v = rng.standard_normal((8192, 8))
    shares = {}
    for off, tau in ((5.0, 3.0), (3.0, 5.0)):
        st = {}
        M.forward(s, v, off=off, tau=tau, stats=st)
        shares[off] = st["redo_rows"] / st["row_tiles"]
    assert shares[5.0] > 0.02 and shares[3.0] < 1e-3

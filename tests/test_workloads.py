"""Seeded input generator: bf16 rounding, workload shapes, RMS norm, row sampling."""
import math

import numpy as np
import pytest
import torch

import workloads as W


def test_bf16_round_to_nearest_even_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(3.0),
        np.array([0.0, -0.0, 1.0, -1.0, 1e-40, 3.0e38, 65504.0, 1.00390625, 1.01171875],
                 np.float32),
        # exact ties: the low 16 bits are 0x8000, so RNE rounds to the even neighbour
        (np.arange(1, 2000, dtype=np.uint32) << np.uint32(16) | np.uint32(0x8000)).view(np.float32)
        [:1000],
    ])
    ours = W.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # widening back is exact
    assert np.array_equal(W.bf16_to_f32(ours),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_bf16_rejects_non_finite():
    with pytest.raises(ValueError):
        W.bf16_bits(np.array([np.nan], np.float32))


def test_workload_table():
    names = [w.name for w in W.WORKLOADS]
    assert names == ["tiny", "1024px", "2048px_t2i_cfg", "2048px_i2i_ref", "ragged_outliers"]
    for w in W.WORKLOADS:
        assert sum(n for _, n in w.segments) == w.Lq == w.Lk
        assert w.scale == float(np.float32(1 / math.sqrt(w.d)))
    assert W.workload("2048px_t2i_cfg").flops == pytest.approx(7.016e12, rel=1e-3)
    assert W.workload("2048px_i2i_ref").flops == pytest.approx(1.361e13, rel=1e-3)


def test_tiny_inputs_deterministic_and_normal():
    w = W.workload("tiny")
    q, k, v = W.make_qkv(w)
    q2, k2, v2 = W.make_qkv(w)
    assert q.shape == (1, 2, 256, 64) and q.dtype == np.uint16
    assert np.array_equal(q, q2) and np.array_equal(k, k2) and np.array_equal(v, v2)
    for x in (q, k, v):
        f = W.bf16_to_f32(x)
        assert abs(f.mean()) < 0.05 and abs(f.std() - 1) < 0.05


def test_rms_norm_bounds_logits():
    # A small workload with the same recipe as the 1024px one.
    w = W.Workload("rms_small", 1, 2, 300, 300, 128, seed=11, rms_norm=True)
    q, k, _ = W.make_qkv(w)
    qf, kf = (W.bf16_to_f32(x).astype(np.float64) for x in (q, k))
    np.testing.assert_allclose(np.sqrt((qf ** 2).mean(-1)), 1.0, atol=2e-2)
    s = w.scale * np.einsum("bhid,bhjd->bhij", qf, kf)
    # Cauchy-Schwarz: |s| <= scale*|q||k| = sqrt(d) up to the bf16 rounding of q, k
    assert np.abs(s).max() <= math.sqrt(128) * (1 + 2 ** -6)


def test_outlier_rows():
    w = W.Workload("outl_small", 1, 3, 500, 500, 64, seed=4, outlier_frac=0.01)
    _, k, _ = W.make_qkv(w)
    norms = np.sqrt((W.bf16_to_f32(k).astype(np.float64) ** 2).sum(-1))
    big = norms > 4 * math.sqrt(64)
    # the same 5 rows are scaled in every head
    assert big.sum(-1).tolist() == [[5, 5, 5]]
    assert np.array_equal(big[0, 0], big[0, 2])


def test_sample_rows():
    w = W.workload("ragged_outliers")
    r = W.sample_rows(w, 0, 5)
    assert len(r) == 256 and np.all(np.diff(r) > 0) and r[-1] == w.Lq - 1
    assert np.array_equal(r, W.sample_rows(w, 0, 5))
    assert not np.array_equal(r, W.sample_rows(w, 0, 6))
    assert np.array_equal(W.sample_rows(W.workload("tiny"), 0, 1), np.arange(256))


def test_e4m3_round_to_nearest_even_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(40.0),
        rng.standard_normal(20000).astype(np.float32) * np.float32(0.01),     # subnormal range
        np.array([0.0, 448.0, 449.0, 1000.0, -1000.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11,
                  1.0625, 1.1875, 240.0, 248.0, 232.0], np.float32),
    ])
    ours = W.e4m3_bits(x)
    xt = torch.from_numpy(np.clip(x, -448, 448))          # torch saturates only via clamp
    ref = xt.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    back = torch.from_numpy(ours.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(W.e4m3_to_f32(ours), back)


def test_quantize_e4m3_per_tensor_scale():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 50)).astype(np.float32) * np.float32(7.0)
    codes, scale = W.quantize_e4m3(x)
    deq = W.e4m3_to_f32(codes) * scale
    assert np.abs(deq).max() <= 448 * scale * (1 + 1e-6)
    np.testing.assert_allclose(deq, x, rtol=2 ** -3, atol=scale * 2.0 ** -9)


def test_e4m3_every_value_and_midpoint():
    # every non-negative finite e4m3 value, and float32 neighbours of every
    # midpoint between consecutive values (ties go to the even code)
    vals = W.e4m3_to_f32(np.arange(0x7F, dtype=np.uint8))
    assert np.array_equal(W.e4m3_bits(vals), np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(W.e4m3_bits(x), ref)
    assert vals[0x7E] == 448.0 and vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6

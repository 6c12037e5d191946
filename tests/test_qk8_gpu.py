"""GPU parity of the e4m3-QK attention forward and its quantising RMS-norm prologue.

Queries and keys come from the seeded generator as bf16 and are quantised per
tensor to e4m3 on the host (scale = amax / 448, round to nearest even); the
oracle evaluates the FP64 definition on the dequantised values (code value x
scale, exact in float64) with the bf16 values.  Tolerance as for the bf16
path: max|err| <= 2e-2 and relative L2 <= 5e-3.  Exact properties (bit
equality with the bf16 kernel where every logit is exact in fp32, scale
folding) are checked bit for bit.  All calls go through the C-ABI library.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import assert_close, to_device, to_host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dit():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_transformer_joint_causal_b300 as lib
    from diffusion_transformer_joint_causal_b300 import build
    build.build()
    lib.create()
    yield lib
    assert lib.get_device_error() == 0


def to_device_e4m3(codes):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).cuda().view(
        torch.float8_e4m3fn)


def quantise(bits):
    """bf16 bits -> (e4m3 codes, per-tensor scale, float64 dequantised values)."""
    codes, s = W.quantize_e4m3(W.bf16_to_f32(bits))
    return codes, s, W.e4m3_to_f32(codes).astype(np.float64) * s


def run_qk8(dit, q8, k8, v, qs, ks, scale):
    import torch
    out = dit.forward_qk8(to_device_e4m3(q8), to_device_e4m3(k8), to_device(v), qs, ks, scale)
    torch.cuda.synchronize()
    return out


SHAPES = [
    # (B, H, Lq, Lk); d = 128
    (1, 1, 1, 1),
    (1, 2, 77, 77),
    (1, 1, 129, 127),
    (1, 2, 300, 129),
    (1, 1, 256, 1),
    (1, 1, 1, 1000),
    (1, 1, 513, 255),
    (1, 3, 1000, 1000),
    (2, 1, 1500, 700),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_every_element(dit, shape):
    B, H, Lq, Lk = shape
    rng = np.random.default_rng(1000 + Lq * 7 + Lk)
    q8, qs, qd = quantise(W.random_bf16(rng, (B, H, Lq, 128)))
    k8, ks, kd = quantise(W.random_bf16(rng, (B, H, Lk, 128)))
    v = W.random_bf16(rng, (B, H, Lk, 128))
    scale = float(np.float32(1 / math.sqrt(128)))
    got = to_host_f64(run_qk8(dit, q8, k8, v, qs, ks, scale))
    want = oracle.attention(qd, kd, W.bf16_to_f32(v).astype(np.float64), scale)
    assert_close(got, want, str(shape))


@pytest.mark.parametrize("name", ["1024px", "2048px_t2i_cfg", "2048px_i2i_ref", "ragged_outliers"])
def test_workload_sampled_rows(dit, name):
    import torch
    w = W.workload(name)
    q, k, v = W.make_qkv(w)
    q8, qs, _ = quantise(q)
    k8, ks, kd = quantise(k)
    del q, k
    out = run_qk8(dit, q8, k8, v, qs, ks, w.scale)
    bh, rows = [], []
    for b in range(w.B):
        for h in range(w.H):
            r = W.sample_rows(w, b, h)
            bh.append(np.full(r.shape, b * w.H + h))
            rows.append(r)
    bh, rows = np.concatenate(bh), np.concatenate(rows)
    sel = out.view(w.B * w.H, w.Lq, w.d)[torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda()]
    got = to_host_f64(sel)
    # only the sampled query rows are dequantised in full
    qd = np.zeros((w.B * w.H, w.Lq, w.d))
    flat_q8 = q8.reshape(w.B * w.H, w.Lq, w.d)
    qd[bh, rows] = W.e4m3_to_f32(flat_q8[bh, rows]).astype(np.float64) * qs
    want = oracle.attention_rows(qd.reshape(w.B, w.H, w.Lq, w.d), kd,
                                 W.bf16_to_f32(v).astype(np.float64), w.scale, bh, rows)
    assert_close(got, want, name)


def _exact_codes(rng, shape):
    # e4m3 values with |x| in [2^-3, 3.75]: every one is a multiple of 2^-6 below
    # 2^8 of them, so each product is a multiple of 2^-12 and any sum of 128
    # products stays below 2^23 of those units: exact in fp32 in any order.
    e = rng.integers(4, 9, shape)            # biased exponent: 2^-3 .. 2^1
    m = rng.integers(0, 8, shape)
    sign = rng.integers(0, 2, shape) << 7
    return (sign | (e << 3) | m).astype(np.uint8)


def test_bit_identical_to_bf16_kernel_when_logits_exact(dit):
    import torch
    rng = np.random.default_rng(31)
    q8 = _exact_codes(rng, (2, 2, 700, 128))
    k8 = _exact_codes(rng, (2, 2, 900, 128))
    v = W.random_bf16(rng, (2, 2, 900, 128))
    scale = 0.02
    a = run_qk8(dit, q8, k8, v, 1.0, 1.0, scale)
    qb = W.bf16_bits(W.e4m3_to_f32(q8))      # e4m3 values are exact in bf16
    kb = W.bf16_bits(W.e4m3_to_f32(k8))
    b = dit.forward(to_device(qb), to_device(kb), to_device(v), scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_scale_folding_is_exact(dit):
    import torch
    rng = np.random.default_rng(32)
    q8, qs, _ = quantise(W.random_bf16(rng, (1, 2, 600, 128), 2.0))
    k8, ks, _ = quantise(W.random_bf16(rng, (1, 2, 800, 128), 2.0))
    v = W.random_bf16(rng, (1, 2, 800, 128))
    a = run_qk8(dit, q8, k8, v, qs, ks, 0.088)
    b = run_qk8(dit, q8, k8, v, qs * 4.0, ks / 4.0, 0.088)    # same product, powers of two
    c = run_qk8(dit, q8, k8, v, 1.0, 1.0, 0.088 * qs * ks)    # folded by the caller
    d = to_host_f64(c)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert_close(d, to_host_f64(a), "folded scale")


def test_large_logits_and_saturated_codes(dit):
    # Codes up to +-448 (0x7E / 0xFE) with a logit spread far beyond exp's
    # fp32 range: needs the running max.
    rng = np.random.default_rng(33)
    q8 = rng.integers(0, 256, (1, 2, 300, 128)).astype(np.uint8)
    k8 = rng.integers(0, 256, (1, 2, 3000, 128)).astype(np.uint8)
    for x in (q8, k8):
        x[(x & 0x7F) == 0x7F] -= 1           # NaN codes -> +-448
    v = W.random_bf16(rng, (1, 2, 3000, 128))
    qs, ks = 0.01, 0.003       # logits of standard deviation ~30 at scale 8
    got = to_host_f64(run_qk8(dit, q8, k8, v, qs, ks, 8.0))
    want = oracle.attention(W.e4m3_to_f32(q8).astype(np.float64) * qs,
                            W.e4m3_to_f32(k8).astype(np.float64) * ks,
                            W.bf16_to_f32(v).astype(np.float64), 8.0)
    assert_close(got, want, "large logits")


def test_deterministic_and_rows_past_lq_untouched(dit):
    import torch
    rng = np.random.default_rng(34)
    q8, qs, _ = quantise(W.random_bf16(rng, (1, 1, 77, 128)))
    k8, ks, _ = quantise(W.random_bf16(rng, (1, 1, 333, 128)))
    v = to_device(W.random_bf16(rng, (1, 1, 333, 128)))
    q8d, k8d = to_device_e4m3(q8), to_device_e4m3(k8)
    buf = torch.full((2 * 77 * 128 + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[: 77 * 128].view(1, 1, 77, 128)
    dit.forward_qk8(q8d, k8d, v, qs, ks, out=out)
    again = dit.forward_qk8(q8d, k8d, v, qs, ks)
    torch.cuda.synchronize()
    assert torch.all(buf[77 * 128:] == 7.0)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


# ----------------------------------------------------------------- quantising prologue

def _check_codes(got, ref, what):
    """got: e4m3 codes from the GPU; ref: the float64 value before rounding.

    Each code must be the e4m3 rounding of ref, except where ref lies within
    the kernel's fp32 rounding (relative 1e-5) of a midpoint between two e4m3
    values: there either neighbour is valid.
    """
    want = W.e4m3_bits(ref.astype(np.float32))
    bad = got != want
    if np.any(bad):
        g = W.e4m3_to_f32(got[bad]).astype(np.float64)
        w_ = W.e4m3_to_f32(want[bad]).astype(np.float64)
        r = ref[bad]
        mid = (g + w_) / 2
        near = np.abs(r - mid) <= 1e-5 * np.maximum(np.abs(r), 2.0 ** -9)
        adjacent = np.abs(got[bad].astype(int) - want[bad].astype(int)) == 1
        assert np.all(near & adjacent), f"{what}: {int((~(near & adjacent)).sum())} codes off"
    return int(bad.sum())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("weighted", [False, True])
def test_rmsnorm_e4m3_codes(dit, d, weighted):
    import torch
    rng = np.random.default_rng(40 + d + weighted)
    rows = 4099                                    # ragged against every grid step
    x = W.random_bf16(rng, (rows, d), 3.0)
    w = W.random_bf16(rng, (d,), 1.5) if weighted else None
    out_scale = float(np.float32(448.0 / math.sqrt(d) / (1.6 if weighted else 1.0)))
    y8 = dit.rmsnorm_e4m3(to_device(x), out_scale, weight=to_device(w) if weighted else None)
    torch.cuda.synchronize()
    got = y8.view(torch.uint8).cpu().numpy()
    ref = oracle.rmsnorm(x, w, 1e-6) * out_scale
    _check_codes(got, ref, f"d={d} weighted={weighted}")


def test_rmsnorm_e4m3_saturates(dit):
    import torch
    rng = np.random.default_rng(45)
    x = W.random_bf16(rng, (1000, 128))
    y8 = dit.rmsnorm_e4m3(to_device(x), 400.0)     # |value| up to ~4500: most saturate
    torch.cuda.synchronize()
    got = y8.view(torch.uint8).cpu().numpy()
    ref = oracle.rmsnorm(x, None, 1e-6) * 400.0
    assert np.all((got & 0x7F) != 0x7F)            # never a NaN code
    assert np.sum((got & 0x7F) == 0x7E) > 10000
    _check_codes(got, np.clip(ref, -448, 448), "saturating")


def test_rmsnorm_e4m3_then_forward_qk8(dit):
    # The e4m3 pipeline on un-normalised inputs: RMS norm + quantise on the GPU,
    # then the e4m3-QK forward; the oracle normalises in float64, rounds to
    # e4m3 on the host, and evaluates the definition on the dequantised values.
    import torch
    w = W.Workload("pipe", 1, 4, 2000, 2000, 128, seed=21)
    q, k, v = W.make_qkv(w)
    s = float(np.float32(math.sqrt(128) / 448))
    inv = float(np.float32(448 / math.sqrt(128)))
    q8 = dit.rmsnorm_e4m3(to_device(q), inv)
    k8 = dit.rmsnorm_e4m3(to_device(k), inv)
    out = dit.forward_qk8(q8, k8, to_device(v), s, s, w.scale)
    torch.cuda.synchronize()
    got = to_host_f64(out)
    qd = W.e4m3_to_f32(W.e4m3_bits((oracle.rmsnorm(q, None, 1e-6) * inv).astype(np.float32)))
    kd = W.e4m3_to_f32(W.e4m3_bits((oracle.rmsnorm(k, None, 1e-6) * inv).astype(np.float32)))
    want = oracle.attention(qd.astype(np.float64) * s, kd.astype(np.float64) * s,
                            W.bf16_to_f32(v).astype(np.float64), w.scale)
    assert_close(got, want, "rmsnorm_e4m3 + forward_qk8")


def test_split_tail_e4m3(dit):
    # fewer work units than CTA pairs: every unit is split over key ranges
    B, H, Lq, Lk = 1, 2, 900, 6000
    assert dit.workspace_size(B, H, Lq, Lk, 128, qk8=True) > 0
    rng = np.random.default_rng(35)
    q8, qs, qd = quantise(W.random_bf16(rng, (B, H, Lq, 128)))
    k8, ks, kd = quantise(W.random_bf16(rng, (B, H, Lk, 128)))
    v = W.random_bf16(rng, (B, H, Lk, 128))
    got = to_host_f64(run_qk8(dit, q8, k8, v, qs, ks, 0.088))
    want = oracle.attention(qd, kd, W.bf16_to_f32(v).astype(np.float64), 0.088)
    assert_close(got, want, "e4m3 split tail")


def test_negative_scale(dit):
    # either sign of the logit scale: against the oracle, and bit for bit
    # against the positive scale with every key code negated (sign bit 0x80)
    import torch
    rng = np.random.default_rng(36)
    q8, qs, qd = quantise(W.random_bf16(rng, (1, 3, 1000, 128)))
    k8, ks, kd = quantise(W.random_bf16(rng, (1, 3, 1300, 128)))
    v = W.random_bf16(rng, (1, 3, 1300, 128))
    a = run_qk8(dit, q8, k8, v, qs, ks, -0.088)
    want = oracle.attention(qd, kd, W.bf16_to_f32(v).astype(np.float64), -0.088)
    assert_close(to_host_f64(a), want, "e4m3 Q/K, negative scale")
    b = run_qk8(dit, q8, k8 ^ np.uint8(0x80), v, qs, ks, 0.088)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))

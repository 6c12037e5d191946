"""GPU parity of the e4m3 Q/K/V attention forward (P rounded to e4m3 before P.V)
and of the per-tensor e4m3 quantisation kernel.

Inputs come from the seeded generator as bf16 and are quantised per tensor on
the host (scale = amax / 448, nearest even); the oracle evaluates the FP64
definition on the dequantised values (code value x scale, exact in float64).

Tolerance, from the arithmetic of the one rounding the path adds to the
definition (every probability rounded to e4m3 for P.V, unit roundoff
u = 2^-4; the row sum adds the unrounded p): the kernel's weights are
p~_j / sum p = w_j (1 + d_j) with |d_j| <= u wherever p~_j is in e4m3's
normal range, so that part of the error is at most u * sum_j w_j |v_jc|.
Keys below the normal range (each under 2^-9 of the row's largest weight)
carry larger relative errors; the bar doubles the normal-range term and adds
an absolute 1e-4 for them (normalising by the sum of the rounded p instead
would give the same form, 2u/(1-u)):

    |o_gpu - o| <= 2u/(1-u) * sum_j w_j |v_jc| + 2^-8 |o| + 1e-4

element by element (2^-8 |o| covers the bf16 output rounding and the fp32
sums).  sum_j w_j |v_jc| is the oracle's attention with |V|.  A numerical
model of the kernel's arithmetic reaches 0.72 of this bound at worst (the
outlier workload) and a relative L2 error of 0.025-0.027 on diffuse rows
(0.016 on the outlier workload), so the aggregate bar is rel L2 <= 4e-2.
Where every probability is exact in e4m3 (one key per row far above the
rest, or all logits equal) the output is checked to the bf16 rounding.
All calls go through the C-ABI library.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import to_device, to_host_f64

pytestmark = pytest.mark.gpu

U = 2.0 ** -4
REL_L2_FP8 = 4e-2


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


def run_fp8(dit, q8, k8, v8, qs, ks, vs, scale, **kw):
    import torch
    out = dit.forward_fp8(to_device_e4m3(q8), to_device_e4m3(k8), to_device_e4m3(v8), qs, ks, vs,
                          scale, **kw)
    torch.cuda.synchronize()
    return out


def assert_fp8_close(got, want, weighted_abs_v, what=""):
    """got, want: outputs; weighted_abs_v: sum_j w_j |v_jc| from the oracle."""
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    bound = 2 * U / (1 - U) * weighted_abs_v + 2.0 ** -8 * np.abs(want) + 1e-4
    worst = float(np.max(err / bound))
    rel = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))
    assert worst <= 1.0 and rel <= REL_L2_FP8, \
        f"{what}: max err/bound {worst:.3f}, rel L2 {rel:.3e}, max|err| {float(err.max()):.3e}"
    return worst, rel


def check_full(got, qd, kd, vd, scale, what):
    want = oracle.attention(qd, kd, vd, scale)
    wabs = oracle.attention(qd, kd, np.abs(vd), scale)
    return assert_fp8_close(got, want, wabs, what)


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
    rng = np.random.default_rng(2000 + Lq * 7 + Lk)
    q8, qs, qd = quantise(W.random_bf16(rng, (B, H, Lq, 128)))
    k8, ks, kd = quantise(W.random_bf16(rng, (B, H, Lk, 128)))
    v8, vs, vd = quantise(W.random_bf16(rng, (B, H, Lk, 128)))
    scale = float(np.float32(1 / math.sqrt(128)))
    got = to_host_f64(run_fp8(dit, q8, k8, v8, qs, ks, vs, scale))
    check_full(got, qd, kd, vd, scale, str(shape))


@pytest.mark.parametrize("name", ["1024px", "2048px_t2i_cfg", "2048px_i2i_ref", "ragged_outliers"])
def test_workload_sampled_rows(dit, name):
    import torch
    w = W.workload(name)
    q, k, v = W.make_qkv(w)
    q8, qs, _ = quantise(q)
    k8, ks, kd = quantise(k)
    v8, vs, vd = quantise(v)
    del q, k, v
    out = run_fp8(dit, q8, k8, v8, qs, ks, vs, w.scale)
    bh, rows = [], []
    for b in range(w.B):
        for h in range(w.H):
            r = W.sample_rows(w, b, h)
            bh.append(np.full(r.shape, b * w.H + h))
            rows.append(r)
    bh, rows = np.concatenate(bh), np.concatenate(rows)
    sel = out.view(w.B * w.H, w.Lq, w.d)[torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda()]
    got = to_host_f64(sel)
    qd = np.zeros((w.B * w.H, w.Lq, w.d))
    flat_q8 = q8.reshape(w.B * w.H, w.Lq, w.d)
    qd[bh, rows] = W.e4m3_to_f32(flat_q8[bh, rows]).astype(np.float64) * qs
    qd = qd.reshape(w.B, w.H, w.Lq, w.d)
    want = oracle.attention_rows(qd, kd, vd, w.scale, bh, rows)
    wabs = oracle.attention_rows(qd, kd, np.abs(vd), w.scale, bh, rows)
    assert_fp8_close(got, want, wabs, name)


E4M3_16 = 0x58     # code of 16.0 (exponent 4 + 7, mantissa 0)


def _random_value_codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] -= 1                     # NaN codes -> +-448
    return c


@pytest.mark.parametrize("Lq,Lk", [(700, 300), (300, 1000), (513, 128)])
def test_one_key_per_row_selects_its_value_row_exactly(dit, Lq, Lk):
    # Key j_c = 16 e_c for one key per column c (spread over every key tile,
    # the last one ragged), every other key zero; query i = 16 e_pi(i).  Row
    # i's logit is 256 * scale for its key and 0 for all others, 92 log2 units
    # apart: its p is 2^3 exactly and every other p rounds to 0 in e4m3 after
    # the running max moves, so o_i = v_scale * v8[j_pi(i)] to the bf16
    # rounding, whichever key tile holds the key.
    rng = np.random.default_rng(51 + Lk)
    d = 128
    keys_of_col = rng.choice(Lk, size=min(d, Lk), replace=False)
    k8 = np.zeros((1, 1, Lk, d), np.uint8)
    k8[0, 0, keys_of_col, np.arange(len(keys_of_col))] = E4M3_16
    cols = rng.integers(0, len(keys_of_col), Lq)
    q8 = np.zeros((1, 1, Lq, d), np.uint8)
    q8[0, 0, np.arange(Lq), cols] = E4M3_16
    v8 = _random_value_codes(rng, (1, 1, Lk, d))
    vs = 0.01
    got = to_host_f64(run_fp8(dit, q8, k8, v8, 1.0, 1.0, vs, 0.25))
    want = W.e4m3_to_f32(v8[0, 0, keys_of_col[cols]]).astype(np.float64) * vs
    # (the other keys keep weights near e^-64, as in the definition)
    assert np.all(np.abs(got[0, 0] - want) <= 2.0 ** -8 * np.abs(want) + 1e-20)


@pytest.mark.parametrize("Lq,Lk", [(300, 1000), (129, 77)])
def test_equal_logits_give_the_mean_of_the_values(dit, Lq, Lk):
    # q = 0: every logit is 0, every p is 2^3 exactly, o = mean_j v_j (fp32
    # sums of exact products); pins every value column and key of the P.V
    # product to its place.
    rng = np.random.default_rng(61 + Lk)
    q8 = np.zeros((1, 2, Lq, 128), np.uint8)
    k8, ks, _ = quantise(W.random_bf16(rng, (1, 2, Lk, 128)))
    v8, vs, vd = quantise(W.random_bf16(rng, (1, 2, Lk, 128)))
    got = to_host_f64(run_fp8(dit, q8, k8, v8, 1.0, ks, vs, 0.088))
    want = np.broadcast_to(vd.mean(axis=2, keepdims=True), got.shape)
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-4 * np.abs(vd).max())


def test_large_logits_and_saturated_codes(dit):
    # Codes up to +-448 with a logit spread far beyond exp's fp32 range: the
    # running max, the max pass and the rescale of O all act.
    rng = np.random.default_rng(63)
    q8 = _random_value_codes(rng, (1, 2, 300, 128))
    k8 = _random_value_codes(rng, (1, 2, 3000, 128))
    v8 = _random_value_codes(rng, (1, 2, 3000, 128))
    qs, ks, vs = 0.01, 0.003, 0.002
    got = to_host_f64(run_fp8(dit, q8, k8, v8, qs, ks, vs, 8.0))
    dq = lambda c, s: W.e4m3_to_f32(c).astype(np.float64) * s
    check_full(got, dq(q8, qs), dq(k8, ks), dq(v8, vs), 8.0, "large logits")


def test_growing_max_across_key_tiles(dit):
    # Keys whose scale grows tile by tile: the running max rises on most key
    # tiles (by more than the lazy threshold on some), exercising the
    # optimistic pass, the max pass and the O rescale in every order.
    rng = np.random.default_rng(64)
    Lk = 1500
    q8, qs, qd = quantise(W.random_bf16(rng, (1, 2, 400, 128)))
    kf = W.bf16_to_f32(W.random_bf16(rng, (1, 2, Lk, 128)))
    kf *= np.repeat(np.linspace(0.2, 3.0, (Lk + 127) // 128), 128)[:Lk][None, None, :, None]
    k8, ks = W.quantize_e4m3(kf)
    kd = W.e4m3_to_f32(k8).astype(np.float64) * ks
    v8, vs, vd = quantise(W.random_bf16(rng, (1, 2, Lk, 128)))
    got = to_host_f64(run_fp8(dit, q8, k8, v8, qs, ks, vs, 0.3))
    check_full(got, qd, kd, vd, 0.3, "growing max")


def test_value_scale_is_applied_exactly(dit):
    import torch
    rng = np.random.default_rng(65)
    q8, qs, _ = quantise(W.random_bf16(rng, (1, 2, 600, 128)))
    k8, ks, _ = quantise(W.random_bf16(rng, (1, 2, 800, 128)))
    v8, vs, _ = quantise(W.random_bf16(rng, (1, 2, 800, 128)))
    a = run_fp8(dit, q8, k8, v8, qs, ks, vs, 0.088)
    b = run_fp8(dit, q8, k8, v8, qs, ks, vs * 4.0, 0.088)     # a power of two: exact
    c = run_fp8(dit, q8, k8, v8, qs * 2.0, ks / 2.0, vs, 0.088)
    assert torch.equal((a.float() * 4.0).to(torch.bfloat16).view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_deterministic_and_rows_past_lq_untouched(dit):
    import torch
    rng = np.random.default_rng(66)
    q8, qs, _ = quantise(W.random_bf16(rng, (1, 1, 77, 128)))
    k8, ks, _ = quantise(W.random_bf16(rng, (1, 1, 333, 128)))
    v8, vs, _ = quantise(W.random_bf16(rng, (1, 1, 333, 128)))
    q8d, k8d, v8d = to_device_e4m3(q8), to_device_e4m3(k8), to_device_e4m3(v8)
    buf = torch.full((2 * 77 * 128 + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[: 77 * 128].view(1, 1, 77, 128)
    dit.forward_fp8(q8d, k8d, v8d, qs, ks, vs, out=out)
    again = dit.forward_fp8(q8d, k8d, v8d, qs, ks, vs)
    torch.cuda.synchronize()
    assert torch.all(buf[77 * 128:] == 7.0)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def test_split_tail_fp8(dit):
    # fewer work units than CTA pairs: every unit is split over key ranges,
    # and the partial row sums carry 1 / v_scale
    B, H, Lq, Lk = 1, 2, 900, 6000
    assert dit.workspace_size(B, H, Lq, Lk, 128, variant=2) > 0
    rng = np.random.default_rng(67)
    q8, qs, qd = quantise(W.random_bf16(rng, (B, H, Lq, 128)))
    k8, ks, kd = quantise(W.random_bf16(rng, (B, H, Lk, 128)))
    v8, vs, vd = quantise(W.random_bf16(rng, (B, H, Lk, 128)))
    got = to_host_f64(run_fp8(dit, q8, k8, v8, qs, ks, vs, 0.088))
    check_full(got, qd, kd, vd, 0.088, "e4m3 split tail")
    unsplit = to_host_f64(run_fp8(dit, q8, k8, v8, qs, ks, vs, 0.088, workspace=None))
    check_full(unsplit, qd, kd, vd, 0.088, "e4m3 unsplit")


# ----------------------------------------------------------------- quantisation kernel

@pytest.mark.parametrize("n", [1, 7, 8, 4099, 1 << 20, (1 << 20) + 5])
def test_quantize_e4m3_bit_exact(dit, n):
    import torch
    rng = np.random.default_rng(70 + n % 97)
    x = W.random_bf16(rng, (n,), 40.0)             # many values saturate at the scale below
    out_scale = float(np.float32(448.0 / 100.0))
    y8 = dit.quantize_e4m3(to_device(x), out_scale)
    torch.cuda.synchronize()
    got = y8.view(torch.uint8).cpu().numpy()
    # the fp32 product of the bf16 value and the scale, then e4m3 rounding
    want = W.e4m3_bits(W.bf16_to_f32(x) * np.float32(out_scale))
    assert np.array_equal(got, want)


def test_quantize_e4m3_small_and_subnormal_values(dit):
    import torch
    # every bf16 value from 2^-16 to 2^9, both signs: subnormal e4m3 codes,
    # rounding ties, saturation at 448
    mags = (2.0 ** np.linspace(-16, 9, 3001)).astype(np.float32)
    x = W.bf16_bits(np.concatenate([mags, -mags, np.zeros(3, np.float32)]))
    y8 = dit.quantize_e4m3(to_device(x), 1.0)
    torch.cuda.synchronize()
    got = y8.view(torch.uint8).cpu().numpy()
    assert np.array_equal(got, W.e4m3_bits(W.bf16_to_f32(x)))


def test_quantize_then_forward_fp8(dit):
    # The e4m3 pipeline on the device: RMS norm + quantise for Q and K, plain
    # quantisation for V, then the forward; the oracle rounds on the host.
    import torch
    w = W.Workload("pipe8", 1, 4, 2000, 2000, 128, seed=22)
    q, k, v = W.make_qkv(w)
    s = float(np.float32(math.sqrt(128) / 448))
    inv = float(np.float32(448 / math.sqrt(128)))
    vmax = float(np.abs(W.bf16_to_f32(v)).max())
    vs = float(np.float32(vmax / 448))
    inv_vs = float(np.float32(1 / vs))
    q8 = dit.rmsnorm_e4m3(to_device(q), inv)
    k8 = dit.rmsnorm_e4m3(to_device(k), inv)
    v8 = dit.quantize_e4m3(to_device(v), inv_vs)
    out = dit.forward_fp8(q8, k8, v8, s, s, vs, w.scale)
    torch.cuda.synchronize()
    got = to_host_f64(out)
    qd = W.e4m3_to_f32(W.e4m3_bits((oracle.rmsnorm(q, None, 1e-6) * inv).astype(np.float32)))
    kd = W.e4m3_to_f32(W.e4m3_bits((oracle.rmsnorm(k, None, 1e-6) * inv).astype(np.float32)))
    vc = W.e4m3_bits(W.bf16_to_f32(v) * np.float32(inv_vs))
    assert np.array_equal(v8.view(torch.uint8).cpu().numpy(), vc)
    check_full(got, qd.astype(np.float64) * s, kd.astype(np.float64) * s,
               W.e4m3_to_f32(vc).astype(np.float64) * vs, w.scale, "quantise + forward_fp8")


def test_million_key_rows_fp8(dit):
    # e4m3 Q/K/V over 2^20 + 77 keys (8193 key tiles, the split tail in 16
    # chunks whose partial row sums carry 1 / v_scale), every eighth row.
    B, H, Lq, Lk, d = 1, 1, 300, (1 << 20) + 77, 128
    assert dit.workspace_size(B, H, Lq, Lk, d, variant=2) > 0
    rng = np.random.default_rng(2401)
    rms = lambda x: x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + np.float32(1e-6))
    q8, qs = W.quantize_e4m3(rms(rng.standard_normal((B, H, Lq, d), dtype=np.float32)))
    k8, ks = W.quantize_e4m3(rms(rng.standard_normal((B, H, Lk, d), dtype=np.float32)))
    v8, vs = W.quantize_e4m3(rng.standard_normal((B, H, Lk, d), dtype=np.float32))
    scale = float(np.float32(1 / math.sqrt(d)))
    got = to_host_f64(run_fp8(dit, q8, k8, v8, qs, ks, vs, scale))
    dq = lambda c, s: W.e4m3_to_f32(c).astype(np.float64) * s
    rows = np.concatenate([np.arange(0, Lq, 8), [Lq - 1]])
    bh = np.zeros_like(rows)
    qd, kd, vd = dq(q8, qs), dq(k8, ks), dq(v8, vs)
    want = oracle.attention_rows(qd, kd, vd, scale, bh, rows)
    wabs = oracle.attention_rows(qd, kd, np.abs(vd), scale, bh, rows)
    assert_fp8_close(got[0, 0][rows], want, wabs, "2^20 keys, e4m3")


def test_negative_scale(dit):
    # either sign of the logit scale: against the oracle under the e4m3-P
    # bound, and bit for bit against the positive scale with negated key codes
    import torch
    rng = np.random.default_rng(68)
    q8, qs, qd = quantise(W.random_bf16(rng, (1, 3, 1000, 128)))
    k8, ks, kd = quantise(W.random_bf16(rng, (1, 3, 1300, 128)))
    v8, vs, vd = quantise(W.random_bf16(rng, (1, 3, 1300, 128)))
    a = run_fp8(dit, q8, k8, v8, qs, ks, vs, -0.088)
    check_full(to_host_f64(a), qd, kd, vd, -0.088, "e4m3 Q/K/V, negative scale")
    b = run_fp8(dit, q8, k8 ^ np.uint8(0x80), v8, qs, ks, vs, 0.088)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))

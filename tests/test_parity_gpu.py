"""GPU parity: the CUDA attention forward against the FP64 oracle.

All calls go through the C-ABI library (via its ctypes binding).  Small and
ragged shapes compare every output element; the four large workloads compare
256 seeded query rows per (batch, head) (always including the last row, so
the ragged tail tile is covered).  Tolerance: max|err| <= 2e-2 and relative
L2 <= 5e-3.  Exact GPU properties (one-hot selection, a single key, run-to-run
determinism) are checked bit for bit.
"""
import math

import numpy as np
import pytest

import workloads as W
from gpu_util import assert_close, oracle_full, oracle_sampled, to_device, to_host_f64

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


def run(dit, q, k, v, scale):
    import torch
    out = dit.forward(to_device(q), to_device(k), to_device(v), scale)
    torch.cuda.synchronize()
    return out


SHAPES = [
    # (B, H, Lq, Lk, d)
    (1, 1, 1, 1, 64),
    (1, 1, 1, 1, 128),
    (1, 2, 77, 77, 128),
    (1, 1, 127, 129, 64),
    (1, 1, 129, 127, 128),
    (2, 3, 129, 300, 64),
    (1, 2, 300, 129, 128),
    (1, 1, 256, 1, 128),
    (1, 1, 1, 1000, 128),
    (1, 1, 513, 255, 128),
    (2, 2, 384, 640, 64),
    (1, 3, 1000, 1000, 128),
    (3, 1, 700, 1500, 64),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_every_element(dit, shape):
    B, H, Lq, Lk, d = shape
    rng = np.random.default_rng(hash(shape) % 2**32)
    q = W.random_bf16(rng, (B, H, Lq, d))
    k = W.random_bf16(rng, (B, H, Lk, d))
    v = W.random_bf16(rng, (B, H, Lk, d))
    scale = float(np.float32(1 / math.sqrt(d)))
    got = to_host_f64(run(dit, q, k, v, scale))
    assert_close(got, oracle_full(q, k, v, scale), str(shape))


def test_tiny_workload_every_row(dit):
    w = W.workload("tiny")
    q, k, v = W.make_qkv(w)
    got = to_host_f64(run(dit, q, k, v, w.scale))
    assert_close(got, oracle_full(q, k, v, w.scale), w.name)


@pytest.mark.parametrize("name", ["1024px", "2048px_t2i_cfg", "2048px_i2i_ref", "ragged_outliers"])
def test_workload_sampled_rows(dit, name):
    w = W.workload(name)
    q, k, v = W.make_qkv(w)
    out = run(dit, q, k, v, w.scale)
    bh, rows = [], []
    for b in range(w.B):
        for h in range(w.H):
            r = W.sample_rows(w, b, h)
            bh.append(np.full(r.shape, b * w.H + h))
            rows.append(r)
    bh, rows = np.concatenate(bh), np.concatenate(rows)
    import torch
    flat = out.view(w.B * w.H, w.Lq, w.d)
    sel = flat[torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda()]
    got = to_host_f64(sel)
    ref = oracle_sampled(q, k, v, w.scale, bh, rows)
    assert_close(got, ref, name)


def test_large_logits_and_long_keys(dit):
    # Logit spread far beyond exp's fp32 range: needs the running max.
    rng = np.random.default_rng(5)
    q = W.random_bf16(rng, (1, 2, 300, 128), 4.0)
    k = W.random_bf16(rng, (1, 2, 5000, 128), 4.0)
    v = W.random_bf16(rng, (1, 2, 5000, 128))
    got = to_host_f64(run(dit, q, k, v, 0.5))
    assert_close(got, oracle_full(q, k, v, 0.5), "large logits")


def test_zero_scale_is_mean(dit):
    rng = np.random.default_rng(6)
    q = W.random_bf16(rng, (1, 2, 200, 64))
    k = W.random_bf16(rng, (1, 2, 333, 64))
    v = W.random_bf16(rng, (1, 2, 333, 64))
    got = to_host_f64(run(dit, q, k, v, 0.0))
    assert_close(got, oracle_full(q, k, v, 0.0), "scale 0")


def test_single_key_returns_value_exactly(dit):
    rng = np.random.default_rng(7)
    q = W.random_bf16(rng, (2, 2, 300, 128), 3.0)
    k = W.random_bf16(rng, (2, 2, 1, 128), 3.0)
    v = W.random_bf16(rng, (2, 2, 1, 128))
    got = to_host_f64(run(dit, q, k, v, 0.09))
    want = np.broadcast_to(W.bf16_to_f32(v).astype(np.float64), got.shape)
    assert np.array_equal(got, want)


def test_one_hot_selection_exact(dit):
    # Q = 64*e_pi(i), K = identity rows: at scale 2 query i has logit 128 for
    # key pi(i) and 0 for every other key, whose weight exp(-128) is 0 in fp32.
    Lk, d = 128, 128
    Lq = 700
    rng = np.random.default_rng(8)
    pi = rng.integers(0, Lk, Lq)
    qf = np.zeros((1, 1, Lq, d), np.float32)
    qf[0, 0, np.arange(Lq), pi] = 64.0
    kf = np.eye(Lk, d, dtype=np.float32)[None, None]
    v = W.random_bf16(rng, (1, 1, Lk, d))
    got = to_host_f64(run(dit, W.bf16_bits(qf), W.bf16_bits(kf), v, 2.0))
    want = W.bf16_to_f32(v).astype(np.float64)[0, 0, pi]
    assert np.array_equal(got[0, 0], want)


def test_constant_values(dit):
    rng = np.random.default_rng(9)
    q = W.random_bf16(rng, (1, 2, 260, 128))
    k = W.random_bf16(rng, (1, 2, 390, 128))
    c = W.random_bf16(rng, (128,))
    v = np.broadcast_to(c, (1, 2, 390, 128)).copy()
    got = to_host_f64(run(dit, q, k, v, 0.088))
    assert_close(got, np.broadcast_to(W.bf16_to_f32(c).astype(np.float64), got.shape), "const V")


def test_key_value_permutation(dit):
    rng = np.random.default_rng(10)
    q = W.random_bf16(rng, (1, 2, 256, 128))
    k = W.random_bf16(rng, (1, 2, 700, 128))
    v = W.random_bf16(rng, (1, 2, 700, 128))
    perm = rng.permutation(700)
    a = to_host_f64(run(dit, q, k, v, 0.088))
    b = to_host_f64(run(dit, q, k[:, :, perm], v[:, :, perm], 0.088))
    assert_close(b, a, "permuted keys")


def test_deterministic_and_stream(dit):
    import torch
    w = W.Workload("det", 1, 4, 1111, 1111, 128, seed=12, rms_norm=True)
    q, k, v = (to_device(x) for x in W.make_qkv(w))
    a = dit.forward(q, k, v, w.scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b = dit.forward(q, k, v, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_output_rows_past_lq_untouched(dit):
    # The kernel computes whole 128-row tiles; rows beyond Lq must not be stored.
    import torch
    rng = np.random.default_rng(11)
    q = to_device(W.random_bf16(rng, (1, 1, 77, 64)))
    k = to_device(W.random_bf16(rng, (1, 1, 77, 64)))
    v = to_device(W.random_bf16(rng, (1, 1, 77, 64)))
    buf = torch.full((2 * 77 * 64 + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[: 77 * 64].view(1, 1, 77, 64)
    dit.forward(q, k, v, 0.125, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[77 * 64:] == 7.0)


# Split tail: the last, partial wave of work units is cut into key ranges whose
# partial results a second kernel merges.  Shapes with fewer units than CTA
# pairs split every unit (2 to 8 ranges); each must match the oracle element by
# element and the unsplit call within the same tolerance.
SPLIT_SHAPES = [
    # (B, H, Lq, Lk, d)
    (1, 1, 700, 4000, 128),
    (1, 3, 1100, 2500, 128),
    (2, 2, 513, 8192, 128),
    (1, 1, 1, 3000, 128),
]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_split_tail_every_element(dit, shape):
    import torch
    B, H, Lq, Lk, d = shape
    assert dit.workspace_size(B, H, Lq, Lk, d) > 0        # the split path is taken
    rng = np.random.default_rng(2000 + Lq + Lk)
    q = W.random_bf16(rng, (B, H, Lq, d))
    k = W.random_bf16(rng, (B, H, Lk, d))
    v = W.random_bf16(rng, (B, H, Lk, d))
    scale = float(np.float32(1 / math.sqrt(d)))
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    split = dit.forward(qd, kd, vd, scale)                  # workspace="auto"
    whole = dit.forward(qd, kd, vd, scale, workspace=None)
    torch.cuda.synchronize()
    got = to_host_f64(split)
    assert_close(got, oracle_full(q, k, v, scale), f"split {shape}")
    assert_close(got, to_host_f64(whole), f"split vs unsplit {shape}")


def test_split_tail_explicit_workspace_and_rows_past_lq(dit):
    # A caller-owned workspace inside a larger buffer; rows past Lq untouched.
    import torch
    B, H, Lq, Lk, d = 1, 2, 300, 5000, 128
    nb = dit.workspace_size(B, H, Lq, Lk, d)
    assert nb > 0
    rng = np.random.default_rng(2100)
    q = W.random_bf16(rng, (B, H, Lq, d))
    k = W.random_bf16(rng, (B, H, Lk, d))
    v = W.random_bf16(rng, (B, H, Lk, d))
    ws = torch.empty(nb + 4096, dtype=torch.uint8, device="cuda")
    buf = torch.full((B * H * Lq * d + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[: B * H * Lq * d].view(B, H, Lq, d)
    scale = float(np.float32(1 / math.sqrt(d)))
    dit.forward(to_device(q), to_device(k), to_device(v), scale, out=out, workspace=ws[16:16 + nb])
    torch.cuda.synchronize()
    assert torch.all(buf[B * H * Lq * d:] == 7.0)
    assert_close(to_host_f64(out), oracle_full(q, k, v, scale), "explicit workspace")


def test_split_tail_short_workspace_runs_unsplit(dit):
    import torch
    B, H, Lq, Lk, d = 1, 1, 700, 4000, 128
    rng = np.random.default_rng(2200)
    q, k, v = (to_device(W.random_bf16(rng, (B, H, L, d))) for L in (Lq, Lk, Lk))
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    a = dit.forward(q, k, v, 0.088, workspace=small)
    b = dit.forward(q, k, v, 0.088, workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_repeated_calls_bit_identical_at_scale(dit):
    # The full 2048x2048 text-to-image workload (split last wave included):
    # every call of a run, and calls on a second stream, give the same bits.
    import torch
    w = W.workload("2048px_t2i_cfg")
    q, k, v = (to_device(x) for x in W.make_qkv(w))
    first = dit.forward(q, k, v, w.scale)
    outs = [dit.forward(q, k, v, w.scale) for _ in range(4)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        outs.append(dit.forward(q, k, v, w.scale))
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), first.view(torch.int16))


def test_many_heads_short_rows(dit):
    # 160 (b,h) pairs of 300 queries against 2100 keys: 160 work units on 74
    # CTA pairs, the last wave's 12 units split in two key ranges, ragged
    # query and key tails.
    B, H, Lq, Lk, d = 2, 80, 300, 2100, 128
    assert dit.workspace_size(B, H, Lq, Lk, d) > 0
    rng = np.random.default_rng(2300)
    q = W.random_bf16(rng, (B, H, Lq, d))
    k = W.random_bf16(rng, (B, H, Lk, d))
    v = W.random_bf16(rng, (B, H, Lk, d))
    scale = float(np.float32(1 / math.sqrt(d)))
    got = to_host_f64(run(dit, q, k, v, scale))
    bh = np.repeat(np.arange(B * H), 8)
    rows = np.tile(np.array([0, 1, 127, 128, 255, 256, 298, 299]), B * H)
    flat = got.reshape(B * H, Lq, d)[bh, rows]
    assert_close(flat, oracle_sampled(q, k, v, scale, bh, rows), "many heads")


def _rms_bf16(rng, shape):
    x = rng.standard_normal(shape, dtype=np.float32)
    x /= np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + np.float32(1e-6))
    return W.bf16_bits(x)


def test_million_key_rows(dit):
    # Rows over 2^20 + 77 keys (8193 key tiles, the last ragged) with the
    # 2048px workloads' RMS-normalised queries and keys: one work unit, whose
    # key range the split tail cuts into 16 chunks; the fp32 row sums and the
    # merge of the chunks are checked on every eighth query row.
    B, H, Lq, Lk, d = 1, 1, 300, (1 << 20) + 77, 128
    assert dit.workspace_size(B, H, Lq, Lk, d) > 0
    rng = np.random.default_rng(2400)
    q = _rms_bf16(rng, (B, H, Lq, d))
    k = _rms_bf16(rng, (B, H, Lk, d))
    v = W.random_bf16(rng, (B, H, Lk, d))
    scale = float(np.float32(1 / math.sqrt(d)))
    got = to_host_f64(run(dit, q, k, v, scale))
    rows = np.concatenate([np.arange(0, Lq, 8), [Lq - 1]])
    bh = np.zeros_like(rows)
    assert_close(got[0, 0][rows], oracle_sampled(q, k, v, scale, bh, rows), "2^20 keys")


# ----------------------------------------------------------------- the literal C-ABI forward
# dit_attn_forward(q, k, v, out, B, H, Lq, Lk, d, scale, stream) itself, with
# raw device pointers and no workspace (the Python forward goes through the
# workspace entry point).

def _forward_literal(dit, qd, kd, vd, scale):
    import torch
    B, H, Lq, d = qd.shape
    Lk = kd.shape[2]
    out = torch.empty_like(qd)
    rc = dit.forward_ptr(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), B, H, Lq,
                         Lk, d, scale, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, dit.status_string(rc)
    torch.cuda.synchronize()
    assert dit.get_device_error() == 0
    return out


def test_literal_forward_tiny_every_element(dit):
    w = W.workload("tiny")
    q, k, v = W.make_qkv(w)
    out = _forward_literal(dit, to_device(q), to_device(k), to_device(v), w.scale)
    assert_close(to_host_f64(out), oracle_full(q, k, v, w.scale), "dit_attn_forward tiny")


def test_literal_forward_ragged_outliers_sampled(dit):
    import torch
    w = W.workload("ragged_outliers")
    q, k, v = W.make_qkv(w)
    out = _forward_literal(dit, to_device(q), to_device(k), to_device(v), w.scale)
    bh = np.repeat(np.arange(w.B * w.H), 256)
    rows = np.concatenate([W.sample_rows(w, b, h) for b in range(w.B) for h in range(w.H)])
    flat = out.view(w.B * w.H, w.Lq, w.d)
    got = to_host_f64(flat[torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda()])
    assert_close(got, oracle_sampled(q, k, v, w.scale, bh, rows), "dit_attn_forward ragged")


# ----------------------------------------------------------------- negative scales
# softmax(scale * q k^T) v is defined for either sign of the scale; with
# scale < 0 the row max of the scaled logits is scale times the row minimum
# of q k^T.

NEG_SHAPES = [(1, 2, 300, 389, 64), (2, 3, 129, 300, 64), (1, 2, 300, 389, 128),
              (1, 3, 1000, 1000, 128), (1, 1, 1, 1, 128)]


@pytest.mark.parametrize("shape", NEG_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_negative_scale_every_element(dit, shape):
    B, H, Lq, Lk, d = shape
    rng = np.random.default_rng(4000 + Lq + Lk + d)
    q = W.random_bf16(rng, (B, H, Lq, d))
    k = W.random_bf16(rng, (B, H, Lk, d))
    v = W.random_bf16(rng, (B, H, Lk, d))
    scale = float(np.float32(-1 / math.sqrt(d)))
    got = to_host_f64(run(dit, q, k, v, scale))
    assert_close(got, oracle_full(q, k, v, scale), f"negative scale {shape}")


@pytest.mark.parametrize("d", [64, 128])
def test_negative_scale_large_logits(dit, d):
    # logit spread far beyond exp's fp32 range, and a ragged key tail
    rng = np.random.default_rng(4100 + d)
    q = W.random_bf16(rng, (1, 2, 300, d), 4.0)
    k = W.random_bf16(rng, (1, 2, 5000, d), 4.0)
    v = W.random_bf16(rng, (1, 2, 5000, d))
    got = to_host_f64(run(dit, q, k, v, -0.5))
    assert_close(got, oracle_full(q, k, v, -0.5), f"negative scale, large logits, d={d}")


@pytest.mark.parametrize("d", [64, 128])
def test_negative_scale_equals_negated_keys(dit, d):
    # q (-k)^T = -(q k^T) exactly (bf16 negation is exact and the products are
    # summed in the same order), so forward(q, k, v, -s) and forward(q, -k, v, s)
    # see identical fp32 logits and must agree bit for bit.
    import torch
    rng = np.random.default_rng(4200 + d)
    q = W.random_bf16(rng, (2, 2, 700, d))
    k = W.random_bf16(rng, (2, 2, 1300, d))
    v = W.random_bf16(rng, (2, 2, 1300, d))
    neg_k = k ^ np.uint16(0x8000)
    a = run(dit, q, k, v, -0.11)
    b = run(dit, q, neg_k, v, 0.11)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_negative_scale_split_tail(dit):
    B, H, Lq, Lk, d = 1, 1, 700, 4000, 128
    assert dit.workspace_size(B, H, Lq, Lk, d) > 0
    rng = np.random.default_rng(4300)
    q = W.random_bf16(rng, (B, H, Lq, d))
    k = W.random_bf16(rng, (B, H, Lk, d))
    v = W.random_bf16(rng, (B, H, Lk, d))
    got = to_host_f64(run(dit, q, k, v, -0.088))
    assert_close(got, oracle_full(q, k, v, -0.088), "negative scale, split tail")

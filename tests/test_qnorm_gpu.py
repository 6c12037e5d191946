"""The attention forward with the query RMS normalisation folded into the
kernel (dit_attn_forward_qnorm), on the GPU.

The 1024x1024 and 2048x2048 workloads normalise Q and K per token and head
before attention (an input reading: the pages do not print the norm).  End to
end on raw, un-normalised inputs: K through dit_attn_rmsnorm, Q's norm folded
into each row's softmax scale inside the attention kernel; compared with the
FP64 oracle's RMS norm of both followed by the oracle's attention (the bf16
bar: max|err| <= 2e-2, rel L2 <= 5e-3), and with the two-call pipeline
dit_attn_rmsnorm(q) + dit_attn_forward_ws under the same bar (the two differ
by the bf16 rounding of the normalised queries, which the fused form skips).
"""
import dataclasses
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


def _pipelines(dit, q, k, v, scale, workspace="auto"):
    """(fused, two-call) outputs for raw device tensors q, k, v."""
    import torch
    kn = dit.rmsnorm(k)
    fused = dit.forward_qnorm(q, kn, v, scale, workspace=workspace)
    qn = dit.rmsnorm(q)
    two = dit.forward(qn, kn, v, scale, workspace=workspace)
    torch.cuda.synchronize()
    return fused, two


def _oracle_end_to_end(qb, kb, vb, scale, bh=None, rows=None):
    qn = oracle.rmsnorm(qb, None, 1e-6)
    kn = oracle.rmsnorm(kb, None, 1e-6)
    vd = W.bf16_to_f32(vb).astype(np.float64)
    if rows is None:
        return oracle.attention(qn, kn, vd, scale)
    return oracle.attention_rows(qn, kn, vd, scale, bh, rows)


SHAPES = [(1, 1, 1, 1), (1, 2, 77, 77), (1, 1, 129, 127), (2, 3, 300, 129), (1, 1, 513, 255),
          (1, 3, 1000, 1000), (1, 1, 700, 4000)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fused_norm_every_element(dit, shape):
    B, H, Lq, Lk = shape
    rng = np.random.default_rng(5000 + Lq + 3 * Lk)
    qb = W.random_bf16(rng, (B, H, Lq, 128), 2.5)      # raw: rows far from unit RMS
    kb = W.random_bf16(rng, (B, H, Lk, 128), 0.4)
    vb = W.random_bf16(rng, (B, H, Lk, 128))
    scale = float(np.float32(1 / math.sqrt(128)))
    fused, two = _pipelines(dit, to_device(qb), to_device(kb), to_device(vb), scale)
    got = to_host_f64(fused)
    assert_close(got, _oracle_end_to_end(qb, kb, vb, scale), f"fused norm {shape}")
    assert_close(got, to_host_f64(two), f"fused vs two-call {shape}")


def test_fused_norm_rows_of_any_size_negative_scale_and_split(dit):
    # query rows whose RMS spans 2^-8 .. 2^8 (the fold must not depend on it),
    # a negative scale, with and without the split tail
    rng = np.random.default_rng(5100)
    B, H, Lq, Lk = 1, 2, 900, 6000
    assert dit.workspace_size(B, H, Lq, Lk, 128, variant=3) > 0       # split tail taken
    qf = rng.standard_normal((B, H, Lq, 128), dtype=np.float32)
    qf *= np.exp2(rng.integers(-8, 9, (B, H, Lq, 1))).astype(np.float32)
    qb = W.bf16_bits(qf)
    kb = W.random_bf16(rng, (B, H, Lk, 128))
    vb = W.random_bf16(rng, (B, H, Lk, 128))
    for scale, ws in ((0.088, "auto"), (-0.11, None)):
        fused, two = _pipelines(dit, to_device(qb), to_device(kb), to_device(vb), scale, ws)
        got = to_host_f64(fused)
        assert_close(got, _oracle_end_to_end(qb, kb, vb, scale), f"scale {scale}")
        assert_close(got, to_host_f64(two), f"fused vs two-call, scale {scale}")


def test_fused_norm_is_scale_free_and_zero_rows(dit):
    # multiplying q by a power of two leaves the normalised queries unchanged;
    # an all-zero query row with eps = 0 weighs its keys alike (the mean of V)
    import torch
    rng = np.random.default_rng(5200)
    qb = W.random_bf16(rng, (1, 2, 300, 128))
    qb[0, 1, 7] = 0
    kb = W.random_bf16(rng, (1, 2, 500, 128))
    vb = W.random_bf16(rng, (1, 2, 500, 128))
    q, k, v = to_device(qb), to_device(kb), to_device(vb)
    a = dit.forward_qnorm(q, k, v, 0.088, eps=0.0)
    b = dit.forward_qnorm(q * 64, k, v, 0.088, eps=0.0)
    torch.cuda.synchronize()
    assert_close(to_host_f64(b), to_host_f64(a), "q x 64")
    mean_v = W.bf16_to_f32(vb).astype(np.float64)[0, 1].mean(axis=0)
    assert np.all(np.abs(to_host_f64(a)[0, 1, 7] - mean_v) <= 2.0 ** -8 * np.abs(mean_v) + 1e-3)


@pytest.mark.parametrize("name", ["2048px_t2i_cfg", "ragged_outliers"])
def test_fused_norm_workload_raw_inputs(dit, name):
    # the workload's seeded draws before any normalisation
    import torch
    w = dataclasses.replace(W.workload(name), rms_norm=False)
    qb, kb, vb = W.make_qkv(w)
    fused, two = _pipelines(dit, to_device(qb), to_device(kb), to_device(vb), w.scale)
    bh = np.repeat(np.arange(w.B * w.H), 64)
    rows = np.concatenate([W.sample_rows(w, b, h)[::4] for b in range(w.B) for h in range(w.H)])
    sel = (torch.from_numpy(bh).cuda(), torch.from_numpy(rows).cuda())
    got = to_host_f64(fused.view(w.B * w.H, w.Lq, w.d)[sel])
    assert_close(got, _oracle_end_to_end(qb, kb, vb, w.scale, bh, rows), name)
    assert_close(got, to_host_f64(two.view(w.B * w.H, w.Lq, w.d)[sel]), f"{name} vs two-call")

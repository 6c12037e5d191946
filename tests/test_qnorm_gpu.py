"""The attention forward with the query RMS normalisation fused into its load
stage (dit_attn_forward_qnorm), on the GPU.

The 1024x1024 and 2048x2048 workloads normalise Q and K per token and head
before attention (an input reading: the pages do not print the norm).  End to
end on raw, un-normalised inputs: K through dit_attn_rmsnorm, Q normalised
inside the attention kernel; compared with the FP64 oracle's RMS norm of both
followed by the oracle's attention (the bf16 bar: max|err| <= 2e-2, rel L2 <=
5e-3), and bit for bit with the two-call pipeline dit_attn_rmsnorm(q) +
dit_attn_forward_ws (the fused pass repeats dit_attn_rmsnorm's arithmetic).
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


def _pipelines(dit, q, k, v, scale, weight=None, workspace="auto"):
    """(fused, two-call) outputs for raw device tensors q, k, v."""
    import torch
    kn = dit.rmsnorm(k)
    fused = dit.forward_qnorm(q, kn, v, scale, q_weight=weight, workspace=workspace)
    qn = dit.rmsnorm(q, weight=weight)
    two = dit.forward(qn, kn, v, scale, workspace=workspace)
    torch.cuda.synchronize()
    return fused, two


def _oracle_end_to_end(qb, kb, vb, scale, weight=None, bh=None, rows=None):
    qn = oracle.rmsnorm(qb, weight, 1e-6)
    kn = oracle.rmsnorm(kb, None, 1e-6)
    vd = W.bf16_to_f32(vb).astype(np.float64)
    if rows is None:
        return oracle.attention(qn, kn, vd, scale)
    return oracle.attention_rows(qn, kn, vd, scale, bh, rows)


SHAPES = [(1, 1, 1, 1), (1, 2, 77, 77), (1, 1, 129, 127), (2, 3, 300, 129), (1, 1, 513, 255),
          (1, 3, 1000, 1000), (1, 1, 700, 4000)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fused_norm_every_element(dit, shape):
    import torch
    B, H, Lq, Lk = shape
    rng = np.random.default_rng(5000 + Lq + 3 * Lk)
    qb = W.random_bf16(rng, (B, H, Lq, 128), 2.5)      # raw: rows far from unit RMS
    kb = W.random_bf16(rng, (B, H, Lk, 128), 0.4)
    vb = W.random_bf16(rng, (B, H, Lk, 128))
    scale = float(np.float32(1 / math.sqrt(128)))
    fused, two = _pipelines(dit, to_device(qb), to_device(kb), to_device(vb), scale)
    assert torch.equal(fused.view(torch.int16), two.view(torch.int16))
    assert_close(to_host_f64(fused), _oracle_end_to_end(qb, kb, vb, scale), f"fused norm {shape}")


def test_fused_norm_weight_negative_scale_and_unsplit(dit):
    import torch
    rng = np.random.default_rng(5100)
    B, H, Lq, Lk = 1, 2, 900, 6000
    assert dit.workspace_size(B, H, Lq, Lk, 128, variant=3) > 0       # split tail taken
    qb = W.random_bf16(rng, (B, H, Lq, 128), 3.0)
    kb = W.random_bf16(rng, (B, H, Lk, 128))
    vb = W.random_bf16(rng, (B, H, Lk, 128))
    wb = W.bf16_bits(rng.uniform(0.5, 1.5, 128).astype(np.float32))
    w = to_device(wb)
    for scale, ws in ((0.088, "auto"), (-0.11, None)):
        fused, two = _pipelines(dit, to_device(qb), to_device(kb), to_device(vb), scale, w, ws)
        assert torch.equal(fused.view(torch.int16), two.view(torch.int16))
        want = _oracle_end_to_end(qb, kb, vb, scale, wb)
        assert_close(to_host_f64(fused), want, f"weighted, scale {scale}")


@pytest.mark.parametrize("name", ["2048px_t2i_cfg", "ragged_outliers"])
def test_fused_norm_workload_raw_inputs(dit, name):
    # the workload's seeded draws before any normalisation
    import torch
    w = dataclasses.replace(W.workload(name), rms_norm=False)
    qb, kb, vb = W.make_qkv(w)
    fused, two = _pipelines(dit, to_device(qb), to_device(kb), to_device(vb), w.scale)
    assert torch.equal(fused.view(torch.int16), two.view(torch.int16))
    bh = np.repeat(np.arange(w.B * w.H), 64)
    rows = np.concatenate([W.sample_rows(w, b, h)[::4] for b in range(w.B) for h in range(w.H)])
    got = to_host_f64(fused.view(w.B * w.H, w.Lq, w.d)[torch.from_numpy(bh).cuda(),
                                                         torch.from_numpy(rows).cuda()])
    assert_close(got, _oracle_end_to_end(qb, kb, vb, w.scale, None, bh, rows), name)

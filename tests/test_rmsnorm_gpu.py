"""GPU parity of the RMS normalisation kernel against the FP64 oracle.

The kernel computes in fp32 and rounds to bf16, so every output must lie
within one bf16 ulp of the FP64 value, and almost all must equal its
round-to-nearest-even; covers d = 64 and 128, ragged row counts, a weight,
in-place use and the full query tensor of the 2048x2048 workload.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import to_device

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


def bits(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check(got_bits, ref):
    got = W.bf16_to_f32(got_bits).astype(np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)     # one bf16 ulp at |ref|
    assert np.all(np.abs(got - ref) <= ulp + 1e-30), np.max(np.abs(got - ref) / ulp)
    exact = np.mean(got_bits == W.bf16_bits(ref.astype(np.float32)))
    assert exact >= 0.99, exact


@pytest.mark.parametrize("rows,d,weighted,inplace", [
    (1, 64, False, False), (3, 128, True, False), (1001, 64, True, True),
    (4097, 128, False, True), (77777, 128, True, False)])
def test_rmsnorm_matches_oracle(dit, rows, d, weighted, inplace):
    rng = np.random.default_rng(rows)
    x = W.random_bf16(rng, (rows, d), 3.0)
    w = W.random_bf16(rng, (d,)) if weighted else None
    xd = to_device(x)
    wd = to_device(w) if weighted else None
    out = dit.rmsnorm(xd, wd, 1e-6, out=xd if inplace else None)
    import torch
    torch.cuda.synchronize()
    check(bits(out), oracle.rmsnorm(x, w, 1e-6))


def test_rmsnorm_full_query_tensor(dit):
    import torch
    w = W.Workload("q_only", 2, 24, 16896, 1, 128, seed=2)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((w.B, w.H, w.Lq, w.d), dtype=np.float32)
    xb = W.bf16_bits(x)
    out = dit.rmsnorm(to_device(xb))
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(w.B * w.H * w.Lq, 4096, replace=False)
    got = bits(out).reshape(-1, 128)[rows]
    check(got, oracle.rmsnorm(xb.reshape(-1, 128)[rows], None, 1e-6))


def test_rmsnorm_then_attention_matches_normalised_workload(dit):
    """Normalising raw bf16 Q/K on the GPU, then attention, matches the oracle
    applied to the same normalised tensors."""
    import torch
    from gpu_util import assert_close, to_host_f64
    rng = np.random.default_rng(9)
    q = W.random_bf16(rng, (1, 3, 700, 128), 2.0)
    k = W.random_bf16(rng, (1, 3, 900, 128), 2.0)
    v = W.random_bf16(rng, (1, 3, 900, 128))
    qn = dit.rmsnorm(to_device(q))
    kn = dit.rmsnorm(to_device(k))
    out = dit.forward(qn, kn, to_device(v), 0.08838834764831845)
    torch.cuda.synchronize()
    ref = oracle.attention(bits(qn).reshape(q.shape), bits(kn).reshape(k.shape), v,
                           float(np.float32(0.08838834764831845)))
    assert_close(to_host_f64(out), ref, "rmsnorm + attention")


def test_host_output_tensors_are_refused_before_any_launch(dit):
    """An output tensor in host memory would reach a kernel as a host pointer;
    every binding that takes ``out`` refuses it (and a wrong dtype) with
    ValueError, and nothing is launched."""
    import torch
    x = torch.randn(64, 128, device="cuda").to(torch.bfloat16)
    with pytest.raises(ValueError):
        dit.rmsnorm(x, out=torch.empty(64, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        dit.rmsnorm(x, out=torch.empty(64, 128, dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError):
        dit.rmsnorm_e4m3(x, 1.0, out=torch.empty(64, 128, dtype=torch.uint8))
    with pytest.raises(ValueError):
        dit.quantize_e4m3(x, 1.0, out=torch.empty(64, 128, dtype=torch.uint8))
    q = x.view(1, 1, 64, 128)
    with pytest.raises(ValueError):
        dit.forward(q, q, q, out=torch.empty(1, 1, 64, 128, dtype=torch.bfloat16))
    torch.cuda.synchronize()
    assert dit.get_device_error() == 0

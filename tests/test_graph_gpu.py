"""CUDA-graph capture of repeated attention calls.

The forward call keeps no per-call device state and never synchronises, so it
can be captured once and replayed.  The pages report CUDA Graphs cutting
1024x1024 latency from 1.823 s to 0.809 s for the Base model (sns.style
article, sixth paragraph); here capture must reproduce the eager results bit
for bit, for both kernels (d = 64 and d = 128).
"""
import math

import numpy as np
import pytest

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
    assert lib.get_device_error() == 0


@pytest.mark.parametrize("shape", [(1, 2, 300, 389, 64), (1, 4, 1100, 1300, 128)],
                         ids=["d64", "d128"])
def test_graph_replay_matches_eager(dit, shape):
    import torch
    B, H, Lq, Lk, d = shape
    rng = np.random.default_rng(21)
    q = to_device(W.random_bf16(rng, (B, H, Lq, d)))
    k = to_device(W.random_bf16(rng, (B, H, Lk, d)))
    v = to_device(W.random_bf16(rng, (B, H, Lk, d)))
    scale = 1 / math.sqrt(d)
    eager = dit.forward(q, k, v, scale)
    outs = [torch.empty_like(q) for _ in range(3)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for o in outs:
                dit.forward(q, k, v, scale, out=o)
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), eager.view(torch.int16))


def test_graph_replay_time_1024px(dit):
    """Eager versus graph replay on the 1024x1024 shape (20 calls each)."""
    import torch
    w = W.workload("1024px")
    q, k, v = (to_device(x) for x in W.make_qkv(w))
    out = torch.empty_like(q)
    n = 20
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(n):
                dit.forward(q, k, v, w.scale, out=out)
    torch.cuda.synchronize()
    ref = dit.forward(q, k, v, w.scale)
    for _ in range(3):
        dit.forward(q, k, v, w.scale, out=out)
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        dit.forward(q, k, v, w.scale, out=out)
    e1.record()
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / n
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    graph_ms = e0.elapsed_time(e1) / n
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    print(f"\n1024px: eager {eager_ms:.4f} ms/call, graph {graph_ms:.4f} ms/call "
          f"({w.flops / graph_ms / 1e9:.0f} TFLOP/s in the graph)")
    assert graph_ms <= eager_ms * 1.05


def test_graph_replay_e4m3_pipeline(dit):
    """The e4m3 path captured as one graph: RMS-norm + e4m3 quantisation of Q
    and K, then the e4m3-QK forward; replays must equal the eager calls bit
    for bit."""
    import torch
    rng = np.random.default_rng(22)
    B, H, L, d = 1, 3, 1000, 128
    q = to_device(W.random_bf16(rng, (B, H, L, d)))
    k = to_device(W.random_bf16(rng, (B, H, L, d)))
    v = to_device(W.random_bf16(rng, (B, H, L, d)))
    s = float(np.float32(math.sqrt(d) / 448))
    inv = float(np.float32(448 / math.sqrt(d)))

    def pipeline(q8, k8, out):
        dit.rmsnorm_e4m3(q, inv, out=q8)
        dit.rmsnorm_e4m3(k, inv, out=k8)
        dit.forward_qk8(q8, k8, v, s, s, out=out)

    e_q8, e_k8, eager = torch.empty_like(q, dtype=torch.float8_e4m3fn), \
        torch.empty_like(k, dtype=torch.float8_e4m3fn), torch.empty_like(q)
    pipeline(e_q8, e_k8, eager)
    q8, k8, out = torch.empty_like(e_q8), torch.empty_like(e_k8), torch.empty_like(q)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            pipeline(q8, k8, out)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(q8.view(torch.uint8), e_q8.view(torch.uint8))
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_graph_replay_fp8_pipeline(dit):
    """The e4m3 Q/K/V path captured as one graph: RMS-norm + quantisation of
    Q and K, quantisation of V, the e4m3 Q/K/V forward with a split tail;
    replays must equal the eager calls bit for bit."""
    import torch
    rng = np.random.default_rng(24)
    B, H, Lq, Lk, d = 1, 2, 900, 6000, 128
    assert dit.workspace_size(B, H, Lq, Lk, d, variant=2) > 0
    q = to_device(W.random_bf16(rng, (B, H, Lq, d)))
    k = to_device(W.random_bf16(rng, (B, H, Lk, d)))
    v = to_device(W.random_bf16(rng, (B, H, Lk, d)))
    s = float(np.float32(math.sqrt(d) / 448))
    inv = float(np.float32(448 / math.sqrt(d)))
    vs = 0.0125

    def pipeline(q8, k8, v8, out):
        dit.rmsnorm_e4m3(q, inv, out=q8)
        dit.rmsnorm_e4m3(k, inv, out=k8)
        dit.quantize_e4m3(v, 1 / vs, out=v8)
        dit.forward_fp8(q8, k8, v8, s, s, vs, out=out)

    def buffers():
        return (torch.empty_like(q, dtype=torch.float8_e4m3fn),
                torch.empty_like(k, dtype=torch.float8_e4m3fn),
                torch.empty_like(v, dtype=torch.float8_e4m3fn), torch.empty_like(q))

    eager = buffers()
    pipeline(*eager)
    captured = buffers()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            pipeline(*captured)
    torch.cuda.synchronize()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(captured[2].view(torch.uint8), eager[2].view(torch.uint8))
    assert torch.equal(captured[3].view(torch.int16), eager[3].view(torch.int16))


def test_graph_replay_split_tail(dit):
    """A call whose work units are split over key ranges (attention kernel,
    then the merge kernel, workspace from the capture's memory pool) replays
    bit for bit."""
    import torch
    B, H, Lq, Lk, d = 1, 2, 900, 6000, 128
    assert dit.workspace_size(B, H, Lq, Lk, d) > 0
    rng = np.random.default_rng(23)
    q, k, v = (to_device(W.random_bf16(rng, (B, H, L, d))) for L in (Lq, Lk, Lk))
    eager = dit.forward(q, k, v, 0.088)
    out = torch.empty_like(q)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            dit.forward(q, k, v, 0.088, out=out)
    torch.cuda.synchronize()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))

"""CUDA-graph capture of repeated attention calls.

The forward call keeps no per-call device state and never synchronises, so it
can be captured once and replayed.  The pages report CUDA Graphs cutting
1024x1024 latency from 1.823 s to 0.809 s for the Base model (sns.style
article, sixth paragraph).  Every replay here is checked twice: against the
FP64 oracle under the tolerance of its path (the bf16 bar for bf16 and e4m3
Q/K, the derived e4m3-P bound for e4m3 Q/K/V), and bit for bit against the
eager calls of the same library.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import assert_close, oracle_full, oracle_sampled, to_device, to_host_f64

pytestmark = pytest.mark.gpu

U = 2.0 ** -4          # e4m3 unit roundoff: the e4m3-P bound (as in test_fp8_gpu)
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


def _capture(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.synchronize()
    return g


def _assert_fp8_close(got, qd, kd, vd, scale, what):
    want = oracle.attention(qd, kd, vd, scale)
    wabs = oracle.attention(qd, kd, np.abs(vd), scale)
    err = np.abs(got - want)
    bound = 2 * U / (1 - U) * wabs + 2.0 ** -8 * np.abs(want) + 1e-4
    rel = float(np.linalg.norm(got - want) / np.linalg.norm(want))
    assert np.all(np.isfinite(got)) and np.all(err <= bound) and rel <= REL_L2_FP8, \
        f"{what}: max err/bound {float(np.max(err / bound)):.3f}, rel L2 {rel:.3e}"


def _e4m3_dequant(t, s):
    import torch
    return W.e4m3_to_f32(t.view(torch.uint8).cpu().numpy()).astype(np.float64) * s


@pytest.mark.parametrize("shape", [(1, 2, 300, 389, 64), (1, 4, 1100, 1300, 128)],
                         ids=["d64", "d128"])
def test_graph_replay_matches_oracle_and_eager(dit, shape):
    import torch
    B, H, Lq, Lk, d = shape
    rng = np.random.default_rng(21)
    qh = W.random_bf16(rng, (B, H, Lq, d))
    kh = W.random_bf16(rng, (B, H, Lk, d))
    vh = W.random_bf16(rng, (B, H, Lk, d))
    q, k, v = to_device(qh), to_device(kh), to_device(vh)
    scale = float(np.float32(1 / math.sqrt(d)))
    eager = dit.forward(q, k, v, scale)
    outs = [torch.empty_like(q) for _ in range(3)]

    def calls():
        for o in outs:
            dit.forward(q, k, v, scale, out=o)

    g = _capture(calls)
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    want = oracle_full(qh, kh, vh, scale)
    for o in outs:
        assert_close(to_host_f64(o), want, f"graph replay {shape}")
        assert torch.equal(o.view(torch.int16), eager.view(torch.int16))


def test_graph_replay_time_1024px(dit):
    """Eager versus graph replay on the 1024x1024 shape (20 calls each); the
    replayed output against the oracle on the seeded 256-row sample per head."""
    import torch
    w = W.workload("1024px")
    qh, kh, vh = W.make_qkv(w)
    q, k, v = to_device(qh), to_device(kh), to_device(vh)
    out = torch.empty_like(q)
    n = 20

    def calls():
        for _ in range(n):
            dit.forward(q, k, v, w.scale, out=out)

    g = _capture(calls)
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
    out.zero_()
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    graph_ms = e0.elapsed_time(e1) / n
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    bh = np.repeat(np.arange(w.B * w.H), 256)
    rows = np.concatenate([W.sample_rows(w, b, h) for b in range(w.B) for h in range(w.H)])
    got = to_host_f64(out.view(w.B * w.H, w.Lq, w.d)[torch.from_numpy(bh).cuda(),
                                                       torch.from_numpy(rows).cuda()])
    assert_close(got, oracle_sampled(qh, kh, vh, w.scale, bh, rows), "1024px graph replay")
    print(f"\n1024px: eager {eager_ms:.4f} ms/call, graph {graph_ms:.4f} ms/call "
          f"({w.flops / graph_ms / 1e9:.0f} TFLOP/s in the graph)")
    assert graph_ms <= eager_ms * 1.05


def test_graph_replay_e4m3_pipeline(dit):
    """The e4m3 path captured as one graph: RMS-norm + e4m3 quantisation of Q
    and K, then the e4m3-QK forward.  The replayed codes are the host's e4m3
    rounding of the FP64 RMS norm, the replayed output meets the bf16 bar
    against the oracle on those codes, and both equal the eager calls."""
    import torch
    rng = np.random.default_rng(22)
    B, H, L, d = 1, 3, 1000, 128
    qh = W.random_bf16(rng, (B, H, L, d))
    kh = W.random_bf16(rng, (B, H, L, d))
    vh = W.random_bf16(rng, (B, H, L, d))
    q, k, v = to_device(qh), to_device(kh), to_device(vh)
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
    g = _capture(lambda: pipeline(q8, k8, out))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(q8.view(torch.uint8), e_q8.view(torch.uint8))
    assert torch.equal(k8.view(torch.uint8), e_k8.view(torch.uint8))
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    for codes, x in ((q8, qh), (k8, kh)):
        host = W.e4m3_bits((oracle.rmsnorm(x, None, 1e-6) * inv).astype(np.float32))
        got = codes.view(torch.uint8).cpu().numpy()
        # a code may differ only where the fp32 value sits on a rounding midpoint
        assert np.count_nonzero(got != host) <= 1e-4 * got.size
    want = oracle.attention(_e4m3_dequant(q8, s), _e4m3_dequant(k8, s),
                            W.bf16_to_f32(vh).astype(np.float64), float(np.float32(1 / math.sqrt(d))))
    assert_close(to_host_f64(out), want, "e4m3 Q/K graph replay")


def test_graph_replay_fp8_pipeline(dit):
    """The e4m3 Q/K/V path captured as one graph: RMS-norm + quantisation of
    Q and K, quantisation of V, the e4m3 Q/K/V forward with a split tail.
    The replayed output meets the e4m3-P bound against the oracle on the
    replayed codes (the V codes are checked bit for bit against the host's
    quantisation) and equals the eager calls."""
    import torch
    rng = np.random.default_rng(24)
    B, H, Lq, Lk, d = 1, 2, 900, 6000, 128
    assert dit.workspace_size(B, H, Lq, Lk, d, variant=2) > 0
    qh = W.random_bf16(rng, (B, H, Lq, d))
    kh = W.random_bf16(rng, (B, H, Lk, d))
    vh = W.random_bf16(rng, (B, H, Lk, d))
    q, k, v = to_device(qh), to_device(kh), to_device(vh)
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
    g = _capture(lambda: pipeline(*captured))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(captured[2].view(torch.uint8), eager[2].view(torch.uint8))
    assert torch.equal(captured[3].view(torch.int16), eager[3].view(torch.int16))
    vc = W.e4m3_bits(W.bf16_to_f32(vh) * np.float32(1 / vs))
    assert np.array_equal(captured[2].view(torch.uint8).cpu().numpy(), vc)
    _assert_fp8_close(to_host_f64(captured[3]), _e4m3_dequant(captured[0], s),
                      _e4m3_dequant(captured[1], s), _e4m3_dequant(captured[2], vs),
                      float(np.float32(1 / math.sqrt(d))), "e4m3 Q/K/V graph replay")


def test_graph_replay_split_tail(dit):
    """A call whose work units are split over key ranges (attention kernel,
    then the merge kernel, workspace from the capture's memory pool): the
    replay meets the bf16 bar against the oracle and equals the eager call."""
    import torch
    B, H, Lq, Lk, d = 1, 2, 900, 6000, 128
    assert dit.workspace_size(B, H, Lq, Lk, d) > 0
    rng = np.random.default_rng(23)
    qh, kh, vh = (W.random_bf16(rng, (B, H, L, d)) for L in (Lq, Lk, Lk))
    q, k, v = to_device(qh), to_device(kh), to_device(vh)
    eager = dit.forward(q, k, v, 0.088)
    out = torch.empty_like(q)
    g = _capture(lambda: dit.forward(q, k, v, 0.088, out=out))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert_close(to_host_f64(out), oracle_full(qh, kh, vh, 0.088), "split tail graph replay")
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_graph_replay_rmsnorm_prologue_pipeline(dit):
    """The RMS-norm prologue pipeline captured as one graph (dit_attn_rmsnorm of
    raw Q and of raw K, then the forward): the replay meets the bf16 bar
    against the oracle's RMS norm + attention and equals the eager calls."""
    import torch
    rng = np.random.default_rng(25)
    B, H, Lq, Lk, d = 1, 3, 1100, 1300, 128
    qh = W.random_bf16(rng, (B, H, Lq, d), 2.0)
    kh = W.random_bf16(rng, (B, H, Lk, d), 0.5)
    vh = W.random_bf16(rng, (B, H, Lk, d))
    q, k, v = to_device(qh), to_device(kh), to_device(vh)
    scale = float(np.float32(1 / math.sqrt(d)))

    def pipeline(qn, kn, out):
        dit.rmsnorm(q, out=qn)
        dit.rmsnorm(k, out=kn)
        dit.forward(qn, kn, v, scale, out=out)

    eager = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(q))
    pipeline(*eager)
    captured = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(q))
    g = _capture(lambda: pipeline(*captured))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(captured[2].view(torch.int16), eager[2].view(torch.int16))
    want = oracle.attention(oracle.rmsnorm(qh, None, 1e-6), oracle.rmsnorm(kh, None, 1e-6),
                            W.bf16_to_f32(vh).astype(np.float64), scale)
    assert_close(to_host_f64(captured[2]), want, "RMS-norm pipeline graph replay")

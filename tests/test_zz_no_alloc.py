"""dit_attn_forward_noalloc: the forward for callers that cannot allocate
device memory while they run (an engine that reserves all memory up front,
code inside an allocator's own callback, a loop that must not enter
cudaMalloc).  Its split-tail scratch is a file-scope device array held by the
library, so that the call allocates nothing.

CPU: the entry point is exported and validates its arguments before any CUDA
call.  GPU: two calls in a row against the caller-workspace entry point (the
same split plan and arithmetic, only the scratch address differs: bit for
bit) and against the FP64 oracle (max|err| <= 2e-2, rel L2 <= 5e-3); no
device memory taken by the call, neither from torch's caching allocator nor
from the CUDA driver; NOT_INITIALIZED before dit_attn_create().

This file is collected last, so that a run stopping at its first failure has
run every other test; it also passes alone in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest

import diffusion_transformer_joint_causal_b300 as dit
import workloads as W
from gpu_util import assert_close, oracle_full, to_device, to_host_f64

A = 0x7f0000000000
MB = 1 << 20


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def test_noalloc_symbol_exported():
    assert hasattr(ctypes.CDLL(dit.library_path()), "dit_attn_forward_noalloc")


@pytest.mark.parametrize("args,expect", [
    ((0, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 128, 0.125), 1),       # null q
    ((A + 8, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 128, 0.125), 1),   # misaligned q
    ((A, A + MB, A + 2 * MB, A + 512, 1, 1, 8, 8, 128, 0.125), 1),          # out overlaps q
    ((A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 96, 0.125), 2),        # d = 96
])
def test_noalloc_rejects_bad_arguments(args, expect):
    assert dit.forward_noalloc_ptr(*args) == expect


@pytest.mark.skipif(_has_gpu(), reason="checks the no-device path")
def test_noalloc_no_device():
    assert dit.forward_noalloc_ptr(A, A + MB, A + 2 * MB, A + 3 * MB, 1, 1, 8, 8, 128, 0.125) == 4


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from diffusion_transformer_joint_causal_b300 import build
    build.build()
    dit.create()
    yield dit
    assert dit.get_device_error() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 1, 700, 4000, 128), (2, 2, 513, 8192, 128),
                                   (1, 2, 300, 389, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_noalloc_parity(lib, shape):
    import torch
    B, H, Lq, Lk, d = shape
    rng = np.random.default_rng(3000 + Lq + Lk)
    q = W.random_bf16(rng, (B, H, Lq, d))
    k = W.random_bf16(rng, (B, H, Lk, d))
    v = W.random_bf16(rng, (B, H, Lk, d))
    scale = float(np.float32(1 / math.sqrt(d)))
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    ws = lib.forward(qd, kd, vd, scale)        # caller workspace, the same split plan
    want = oracle_full(q, k, v, scale)
    # two calls in a row share the scratch; the second must not see the first's leftovers
    for call in range(2):
        out = torch.full_like(qd, float("nan"))
        lib.forward_noalloc(qd, kd, vd, out, scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ws.view(torch.int16)), f"call {call}"
        assert_close(to_host_f64(out), want, f"noalloc {shape} call {call}")


@pytest.mark.gpu
def test_noalloc_large_split_workload_allocates_nothing(lib):
    # 2048px image-to-image: the last wave's 6 units run as 72 key-range chunks
    # (19 MB of scratch, inside the library's array).
    import torch
    w = W.workload("2048px_i2i_ref")
    assert 0 < lib.workspace_size(w.B, w.H, w.Lq, w.Lk, w.d) <= 80 * 512 * 130 * 4
    q, k, v = (to_device(x) for x in W.make_qkv(w))
    outs = [torch.empty_like(q) for _ in range(2)]
    ref = lib.forward(q, k, v, w.scale)
    lib.forward_noalloc(q, k, v, outs[0], w.scale)     # warm: module and kernels loaded
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    for o in outs:
        lib.forward_noalloc(q, k, v, o, w.scale)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before     # the CUDA driver's view: nothing taken
    assert torch.cuda.memory_allocated() == torch_before
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


@pytest.mark.gpu
def test_noalloc_needs_create(lib):
    import torch
    q = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lib.destroy()
    try:
        rc = lib.forward_noalloc_ptr(q.data_ptr(), q.data_ptr(), q.data_ptr(), out.data_ptr(),
                                     1, 1, 8, 8, 128, 0.125)
        assert rc == 3                                 # NOT_INITIALIZED
    finally:
        lib.create()
    out2 = lib.forward_noalloc(q, q, q, out)
    torch.cuda.synchronize()
    assert torch.equal(out2.float(), torch.zeros_like(out2.float()))

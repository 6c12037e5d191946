"""dit_attn_forward_noalloc: the forward whose split-tail scratch is a
file-scope device array held by the library, so that the call allocates
nothing.

CPU: the entry point is exported and validates its arguments before any CUDA
call.  GPU: parity with the FP64 oracle on shapes whose work units are split
over key ranges, bit equality with the caller-workspace entry point (the same
split plan and arithmetic, only the scratch address differs), and no device
memory allocated by the call.
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
    out = torch.empty_like(qd)
    lib.forward_noalloc(qd, kd, vd, out, scale)
    ws = lib.forward(qd, kd, vd, scale)        # caller workspace, the same split plan
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ws.view(torch.int16))
    assert_close(to_host_f64(out), oracle_full(q, k, v, scale), f"noalloc {shape}")


@pytest.mark.gpu
def test_noalloc_large_split_workload_allocates_nothing(lib):
    # 2048px image-to-image: the last wave's 6 units run as 72 key-range chunks
    # (19 MB of scratch, inside the library's array).
    import torch
    w = W.workload("2048px_i2i_ref")
    assert 0 < lib.workspace_size(w.B, w.H, w.Lq, w.Lk, w.d) <= 80 * 512 * 130 * 4
    q, k, v = (to_device(x) for x in W.make_qkv(w))
    out = torch.empty_like(q)
    ref = lib.forward(q, k, v, w.scale)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    lib.forward_noalloc(q, k, v, out, w.scale)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))

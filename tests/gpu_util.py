"""Shared helpers for the GPU tests: device upload of bf16 bit arrays and the
parity comparison against the FP64 oracle."""
import numpy as np

import oracle
from workloads import bf16_to_f32

# Tolerance for the bf16 attention output against the FP64 definition:
# max |err| <= 2e-2 and relative L2 <= 5e-3 over all compared elements.
MAX_ABS = 2e-2
REL_L2 = 5e-3


def to_device(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_host_f64(t) -> np.ndarray:
    import torch
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return bf16_to_f32(bits).astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    return max_abs, rel


def assert_close(got, ref, what=""):
    max_abs, rel = errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max|err| {max_abs:.3e} rel L2 {rel:.3e}"
    return max_abs, rel


def oracle_full(q, k, v, scale):
    return oracle.attention(q, k, v, scale)


def oracle_sampled(q, k, v, scale, bh, rows):
    return oracle.attention_rows(q, k, v, scale, bh, rows)

"""Seeded synthetic inputs for the joint text+image attention forward.

This module is shared by the CUDA path (tests, bench, smoke) and by the FP64
oracle's tests.  It holds no attention arithmetic: it only draws random
numbers, applies the per-token RMS normalisation that some workloads ask for,
and rounds float32 to bfloat16 bit patterns.

Workloads (shapes follow the FLUX-3-Image-Klein-class DiT of "Speed Up Image
Generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs", Key takeaways,
second item: denoising dominates at 2048x2048 and dense BF16 attention takes
about 60% of DiT kernel time; 1024x1024 and 2048x2048 text-to-image and
image-to-image are the pages' workloads).  The head count, head dim and token
counts are not printed on the pages; they are the stated workload sizes:

  tiny            B=1 H=2  L=256   (64 text + 192 image)           d=64   N(0,1)
  1024px          B=1 H=24 L=4608  (4096 image + 512 text)         d=128  N(0,1), Q/K RMS-normed
  2048px_t2i_cfg  B=2 H=24 L=16896 (16384 image + 512 text)        d=128  as 1024px
  2048px_i2i_ref  B=1 H=24 L=33280 (16384+16384 ref + 512 text)    d=128  as 1024px
  ragged_outliers B=1 H=24 L=9549  (9216 + 333)                    d=128  N(0,1), 1% key rows x8

Recipe (every workload): rng = numpy.random.default_rng(seed); q, k, v are
three successive rng.standard_normal((B,H,L,d), float32) draws.  Optional RMS
norm of q and k over d with eps 1e-6 in float32.  Optional outliers: after the
v draw, rng.choice(L, round(frac*L), replace=False) picks key rows that are
multiplied by 8 in every (b,h).  Finally round-to-nearest-even to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "bf16_bits", "bf16_to_f32",
    "make_qkv", "sample_rows", "attention_flops", "e4m3_bits", "e4m3_to_f32",
    "quantize_e4m3",
]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Lq: int
    Lk: int
    d: int
    seed: int
    rms_norm: bool = False
    outlier_frac: float = 0.0
    outlier_gain: float = 8.0
    segments: tuple = field(default_factory=tuple)   # (label, tokens) of the joint sequence
    sampled_rows: int = 0    # 0: the oracle checks every row; else rows per (b,h)

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d), as the float32 value the GPU receives."""
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def flops(self) -> float:
        return attention_flops(self.B, self.H, self.Lq, self.Lk, self.d)


WORKLOADS = [
    Workload("tiny", 1, 2, 256, 256, 64, seed=0,
             segments=(("text", 64), ("image", 192))),
    Workload("1024px", 1, 24, 4608, 4608, 128, seed=1, rms_norm=True,
             segments=(("image", 4096), ("text", 512)), sampled_rows=256),
    Workload("2048px_t2i_cfg", 2, 24, 16896, 16896, 128, seed=2, rms_norm=True,
             segments=(("image", 16384), ("text", 512)), sampled_rows=256),
    Workload("2048px_i2i_ref", 1, 24, 33280, 33280, 128, seed=3, rms_norm=True,
             segments=(("target", 16384), ("reference", 16384), ("text", 512)),
             sampled_rows=256),
    Workload("ragged_outliers", 1, 24, 9549, 9549, 128, seed=4, outlier_frac=0.01,
             segments=(("image", 9216), ("text", 333)), sampled_rows=256),
]


def workload(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def attention_flops(B, H, Lq, Lk, d) -> float:
    """Dense attention forward work: 2*Lq*Lk*d for QK^T plus the same for PV."""
    return 4.0 * B * H * Lq * Lk * d


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite input")
    u = x.view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_table() -> np.ndarray:
    """Values of the 127 non-negative finite e4m3 codes 0x00..0x7E (bias 7, no inf)."""
    codes = np.arange(0x7F, dtype=np.int64)
    e, m = codes >> 3, codes & 7
    return np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))


_E4M3 = _e4m3_table()


def e4m3_to_f32(codes: np.ndarray) -> np.ndarray:
    """Widen e4m3 codes (uint8; 0x7F/0xFF NaN are not produced here) to float32."""
    c = np.ascontiguousarray(codes, dtype=np.uint8).astype(np.int64)
    mag = _E4M3[np.minimum(c & 0x7F, 0x7E)]
    return np.where(c & 0x80, -mag, mag).astype(np.float32)


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to e4m3 (nearest, ties to even; saturate at 448; sign kept on zero)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite input")
    a = np.minimum(np.abs(x), np.float32(448.0))
    u = a.view(np.uint32)
    # normal binades: keep 3 of float32's 23 mantissa bits (ties to even), rebias 127 -> 7
    normal = ((u + np.uint32(0x7FFFF) + ((u >> np.uint32(20)) & np.uint32(1))) >> np.uint32(20)) \
        - np.uint32((127 - 7) << 3)
    # below 2^-6 the spacing is 2^-9 and the code is the multiple of it
    sub = np.rint(a * np.float32(512.0)).astype(np.uint32)
    code = np.where(a < np.float32(2.0 ** -6), sub, normal).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def quantize_e4m3(x: np.ndarray):
    """Per-tensor e4m3 quantisation: scale = amax / 448, codes = e4m3(x / scale)."""
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    scale = float(np.float32(amax / 448.0)) if amax > 0 else 1.0
    return e4m3_bits(np.asarray(x, np.float32) / np.float32(scale)), scale


def _rms_normalise(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=np.float32)
    return (x / np.sqrt(ms + np.float32(eps))).astype(np.float32)


def make_qkv(w: Workload):
    """Return (q, k, v) as uint16 bf16 bit arrays: q [B,H,Lq,d], k/v [B,H,Lk,d]."""
    rng = np.random.default_rng(w.seed)
    q = rng.standard_normal((w.B, w.H, w.Lq, w.d), dtype=np.float32)
    if w.rms_norm:
        q = _rms_normalise(q)
    qb = bf16_bits(q)
    del q
    k = rng.standard_normal((w.B, w.H, w.Lk, w.d), dtype=np.float32)
    v = rng.standard_normal((w.B, w.H, w.Lk, w.d), dtype=np.float32)
    vb = bf16_bits(v)
    del v
    if w.rms_norm:
        k = _rms_normalise(k)
    if w.outlier_frac > 0.0:
        n_out = int(round(w.outlier_frac * w.Lk))
        idx = rng.choice(w.Lk, n_out, replace=False)
        k[:, :, idx, :] *= np.float32(w.outlier_gain)
    kb = bf16_bits(k)
    return qb, kb, vb


def sample_rows(w: Workload, b: int, h: int, n: int | None = None) -> np.ndarray:
    """Sorted query rows the oracle checks for (b, h); the last row is always in."""
    n = w.sampled_rows if n is None else n
    if n <= 0 or n >= w.Lq:
        return np.arange(w.Lq, dtype=np.int64)
    rows = np.random.default_rng([w.seed, b, h]).choice(w.Lq, n, replace=False)
    if (w.Lq - 1) not in rows:
        rows[-1] = w.Lq - 1
    return np.sort(rows).astype(np.int64)


def random_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """Plain N(0, std^2) bf16 bits for ad-hoc test shapes."""
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))

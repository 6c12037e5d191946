"""FP64 CPU oracle for the dense, non-causal softmax attention forward.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product (the CUDA library and its
binding) never imports this package, and this package never imports the
product: the two share only the seeded input generator in ``workloads``.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, libm
``exp``, no fast-math); this module compiles it with gcc on first use and
marshals numpy arrays through ctypes.  What it computes is the textbook
definition of standard attention (the dense BF16 attention that "Speed Up
Image Generation with FLUX 3 Image Klein on NVIDIA Blackwell GPUs", Key
takeaways, second item, measures): o_i = sum_j softmax_j(scale * q_i . k_j) v_j.

It also holds the RMS normalisation of queries and keys (``rmsnorm``) that the
normalised workloads apply before attention.

Pins (tests/test_oracle_pins.py, tests/test_rmsnorm_oracle.py) tie it to things other than itself: a
50-digit decimal brute force on tiny inputs, the two-key sigmoid closed form,
exact special cases (constant V, Lk = 1, scale = 0, one-hot selection), key /
query permutation equivariance, key-shift invariance and the convex-hull bound.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "libattn_oracle.so")
_lock = threading.Lock()
_lib = None

KIND_BF16 = 0
KIND_F64 = 1


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into libattn_oracle.so (gcc, -O2, no fast-math)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            f = lib.oracle_attention_rows
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                          ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                          ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            g = lib.oracle_rmsnorm
            g.restype = ctypes.c_int
            g.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                          ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]
            _lib = lib
    return _lib


def _prep(x: np.ndarray):
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), KIND_BF16
    return np.ascontiguousarray(x, dtype=np.float64), KIND_F64


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def attention_rows(q, k, v, scale: float, bh, rows, n_threads: int | None = None,
                   return_probs: bool = False):
    """Attention output for the requested (flat head, query row) pairs.

    q: [B,H,Lq,d], k/v: [B,H,Lk,d], all uint16 bf16 bit patterns or all
    float64.  ``scale`` is used as the double given (pass the float32 value the
    GPU receives, widened).  Returns float64 [n, d] (and [n, Lk] probabilities
    p_j / l when ``return_probs``).
    """
    q, kq = _prep(q)
    k, kk = _prep(k)
    v, kv = _prep(v)
    if not (kq == kk == kv):
        raise TypeError("q, k, v must share one element type")
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("expected [B,H,L,d] tensors")
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    if k.shape != (B, H, Lk, d) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    bh = np.ascontiguousarray(bh, dtype=np.int64).ravel()
    rows = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    if bh.shape != rows.shape:
        raise ValueError("bh and rows must have the same length")
    n = rows.size
    out = np.empty((n, d), dtype=np.float64)
    probs = np.empty((n, Lk), dtype=np.float64) if return_probs else None
    nt = default_threads() if n_threads is None else int(n_threads)
    rc = _load().oracle_attention_rows(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, kq, B * H, Lq, Lk, d, float(scale),
        bh.ctypes.data, rows.ctypes.data, n, out.ctypes.data,
        probs.ctypes.data if probs is not None else None, nt)
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return (out, probs) if return_probs else out


def attention(q, k, v, scale: float, n_threads: int | None = None,
              return_probs: bool = False):
    """Every output row: float64 [B,H,Lq,d] (and [B,H,Lq,Lk] probabilities)."""
    B, H, Lq, d = np.shape(q)
    Lk = np.shape(k)[2]
    bh = np.repeat(np.arange(B * H, dtype=np.int64), Lq)
    rows = np.tile(np.arange(Lq, dtype=np.int64), B * H)
    res = attention_rows(q, k, v, scale, bh, rows, n_threads, return_probs)
    if return_probs:
        o, p = res
        return o.reshape(B, H, Lq, d), p.reshape(B, H, Lq, Lk)
    return res.reshape(B, H, Lq, d)


def rmsnorm(x, weight=None, eps: float = 1e-6):
    """y = x / sqrt(mean(x^2 over the last axis) + eps) * weight, float64.

    x: [..., d] uint16 bf16 bits or float64; weight: [d] of the same kind or None.
    """
    x, kx = _prep(x)
    shape = x.shape
    d = shape[-1]
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    w = None
    if weight is not None:
        w, kw = _prep(weight)
        if kw != kx or w.shape != (d,):
            raise ValueError("weight must be [d] of the same element type as x")
    y = np.empty(shape, dtype=np.float64)
    rc = _load().oracle_rmsnorm(x.ctypes.data, w.ctypes.data if w is not None else None, kx,
                                rows, d, float(eps), y.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_rmsnorm rejected its arguments")
    return y

"""Numerical model of the arithmetic of the e4m3-probability attention forward.

Test infrastructure: it restates, in float64 numpy, the steps the e4m3 Q/K/V
kernel takes for one row of logits, so that the tolerance its GPU tests use
can be derived and checked on the CPU.  Per 128-key tile, against a running
max m (log2 units) kept lazily:

  * first tile: m = tile max; p = e4m3(2^(x - m + off));
  * later tiles: p = e4m3(2^(x - m + off)) with the stale m; if the fp32 sum
    of p over either half of the tile (keys 0-63 or 64-127: what one thread
    of the kernel holds) reaches 448 (a value may have saturated), take the
    tile max, rescale l and O by 2^(m - m_tile) when it rose by more than
    tau, and recompute p;
  * l += sum of the unrounded p, O += sum of the rounded p times v;
  * o = O / l, rounded to bf16.

The logits are given in natural units (s = scale * q.k); x = s * log2(e).
"""
import math

import numpy as np

import workloads as W

_E4M3 = W.e4m3_to_f32(np.arange(256, dtype=np.uint8)).astype(np.float64)


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Non-negative values rounded to e4m3 (nearest even, saturating at 448)."""
    return _E4M3[W.e4m3_bits(np.minimum(x, 448.0).astype(np.float32))]


def forward(s: np.ndarray, v: np.ndarray, off: float = 3.0, tau: float = 5.0,
            limit: float = 448.0, bn: int = 128, stats: dict | None = None) -> np.ndarray:
    """Model output for logits s [R, L] (natural units) and values v [L, d]."""
    x = s / math.log(2.0)
    R, L = x.shape
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    O = np.zeros((R, v.shape[1]))
    redo_rows = 0
    for j0 in range(0, L, bn):
        xt = x[:, j0:j0 + bn]
        if j0 == 0:
            m = xt.max(1)
            pr = np.exp2(xt - m[:, None] + off)
        else:
            pr = np.exp2(xt - m[:, None] + off)
            h = bn // 2
            redo = ~((pr[:, :h].sum(1) < limit) & (pr[:, h:].sum(1) < limit))
            if redo.any():
                redo_rows += int(redo.sum())
                mt = xt.max(1)
                grow = redo & (mt > m + tau)
                f = np.where(grow, np.exp2(m - mt), 1.0)
                l *= f
                O *= f[:, None]
                m = np.where(grow, mt, m)
                pr = np.where(redo[:, None], np.exp2(xt - m[:, None] + off), pr)
        l += pr.sum(1)
        O += e4m3_round(pr) @ v[j0:j0 + bn]
    if stats is not None:
        stats["redo_rows"] = redo_rows
        stats["row_tiles"] = R * max(0, (L + bn - 1) // bn - 1)
    o = O / l[:, None]
    return W.bf16_to_f32(W.bf16_bits(o.astype(np.float32))).astype(np.float64)


def bound(weighted_abs_v: np.ndarray, ref: np.ndarray, u: float = 2.0 ** -4) -> np.ndarray:
    """The per-element tolerance of the e4m3-P path (sum_j w_j |v_jc| given)."""
    return 2 * u / (1 - u) * weighted_abs_v + 2.0 ** -8 * np.abs(ref) + 1e-4

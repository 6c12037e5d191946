"""Numerical model of the arithmetic of the bf16-probability attention forward.

Test infrastructure: it restates, in float64 numpy, the per-tile steps of the
bf16 pair kernel's softmax for one row of logits, so that the choice of its
row sum can be checked on the CPU.  Per 128-key tile, against a running max m
(log2 units) kept lazily:

  * first tile: m = tile max; p = 2^(x - m);
  * later tiles: p against the stale m; if the sum of the bf16-rounded p over
    either half of the tile (keys 0-63 or 64-127: what one thread of the
    kernel holds) exceeds 2^48, take the tile max, rescale l and O by
    2^(m - m_tile) when it rose by more than 8, and recompute p;
  * O += bf16(p) times v; l += the bf16-rounded p (rounded_sum) or the fp32 p;
  * o = O / l, rounded to bf16.

The logits are given in natural units (s = scale * q.k); x = s * log2(e).
"""
import math

import numpy as np

import workloads as W


def bf16_round(x: np.ndarray) -> np.ndarray:
    return W.bf16_to_f32(W.bf16_bits(x.astype(np.float32))).astype(np.float64)


def forward(s: np.ndarray, v: np.ndarray, rounded_sum: bool = True, tau: float = 8.0,
            limit: float = 2.0 ** 48, bn: int = 128, stats: dict | None = None) -> np.ndarray:
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
            pr = np.exp2(xt - m[:, None])
        else:
            pr = np.exp2(xt - m[:, None])
            pb, h = bf16_round(pr), bn // 2
            redo = ~((pb[:, :h].sum(1) <= limit) & (pb[:, h:].sum(1) <= limit))
            if redo.any():
                redo_rows += int(redo.sum())
                mt = xt.max(1)
                grow = redo & (mt > m + tau)
                f = np.where(grow, np.exp2(m - mt), 1.0)
                l *= f
                O *= f[:, None]
                m = np.where(grow, mt, m)
                pr = np.where(redo[:, None], np.exp2(xt - m[:, None]), pr)
        pb = bf16_round(pr)
        l += (pb if rounded_sum else pr).sum(1)
        O += pb @ v[j0:j0 + bn]
    if stats is not None:
        stats["redo_rows"] = redo_rows
        stats["row_tiles"] = R * max(0, (L + bn - 1) // bn - 1)
    return bf16_round(O / l[:, None])

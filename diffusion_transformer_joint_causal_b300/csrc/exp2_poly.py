"""Coefficients of the polynomial exp2 that the softmax evaluates on the FMA
pipe for part of its probabilities (exp2_fma in ptx.cuh).

Method: Cody-Waite range reduction (W. J. Cody and W. Waite, "Software Manual
for the Elementary Functions", 1980): 2^x = 2^j * 2^f with j = rint(x) and
f = x - j in [-1/2, 1/2]; 2^f is replaced by the polynomial p(f) of degree n
that minimises the largest relative error max |p(f) / 2^f - 1| over
[-1/2, 1/2], found with the Remez exchange algorithm (E. Remez, 1934): solve
p(f_i) - 2^f_i = (-1)^i E 2^f_i on n + 2 reference points, move the points to
the extrema of the error, repeat until the extrema are level.

    python -m diffusion_transformer_joint_causal_b300.csrc.exp2_poly

prints, for degrees 2 and 3, the coefficients (lowest order first) rounded to
fp32 and the largest relative error of the fp32-rounded polynomial on a dense
grid.  The values are copied into ptx.cuh; tests/test_exp2_poly.py re-derives
them and checks that they agree.
"""
from __future__ import annotations

import numpy as np

LO, HI = -0.5, 0.5


def _rel_err(c, f):
    return np.polynomial.polynomial.polyval(f, c) / np.exp2(f) - 1.0


def remez(n: int, iters: int = 50) -> np.ndarray:
    """Minimax (relative error) coefficients of degree n for 2^f on [LO, HI]."""
    k = np.arange(n + 2)
    pts = (LO + HI) / 2 + (HI - LO) / 2 * -np.cos(np.pi * k / (n + 1))   # Chebyshev extrema
    grid = np.linspace(LO, HI, 200001)
    c = None
    for _ in range(iters):
        # unknowns c_0..c_n, E:  sum_m c_m f_i^m - (-1)^i E 2^f_i = 2^f_i
        A = np.zeros((n + 2, n + 2))
        for m in range(n + 1):
            A[:, m] = pts ** m
        A[:, n + 1] = -((-1.0) ** k) * np.exp2(pts)
        sol = np.linalg.solve(A, np.exp2(pts))
        c = sol[: n + 1]
        e = _rel_err(c, grid)
        # new reference: the extreme of the error on each interval of constant sign
        sign_change = np.nonzero(np.diff(np.sign(e)))[0]
        bounds = np.concatenate([[0], sign_change + 1, [grid.size]])
        ext = [s + int(np.argmax(np.abs(e[s:t]))) for s, t in zip(bounds[:-1], bounds[1:])]
        if len(ext) != n + 2:
            break
        new = grid[ext]
        if np.allclose(new, pts, atol=1e-12):
            pts = new
            break
        pts = new
    return c


def fp32_coefficients(n: int) -> np.ndarray:
    return np.array(remez(n), dtype=np.float32)


def max_rel_error_fp32(c32: np.ndarray) -> float:
    """Largest relative error of Horner's rule in fp32 over f in [-1/2, 1/2]
    (each step rounded to fp32, as the fused multiply-adds do)."""
    f = np.linspace(LO, HI, 400001).astype(np.float32)
    p = np.full_like(f, c32[-1])
    for cm in c32[-2::-1]:
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(cm)).astype(np.float32)
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)))


if __name__ == "__main__":
    for n in (2, 3):
        c = fp32_coefficients(n)
        print(f"degree {n}: " + ", ".join(f"{float(x)!r}f" for x in c)
              + f"   max rel err (fp32 Horner) {max_rel_error_fp32(c):.3e}")

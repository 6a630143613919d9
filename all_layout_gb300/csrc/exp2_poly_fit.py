"""Coefficients of the polynomial 2^f on [0, 1] used by exp2_poly_x2 (ptx.cuh).

The kernel computes part of the softmax exponentials 2^x on the FMA pipe
instead of the MUFU unit: x = n + f with n = floor(x) and f in [0, 1) (a
Cody-Waite style range reduction; one split is exact here because n is an
integer and x has fewer than 24 significant bits above 2^-17), 2^f from a
degree-3 polynomial, and 2^n added into the exponent field.

The polynomial minimises the maximum RELATIVE error |p(f) / 2^f - 1| over
[0, 1]: Remez's exchange algorithm with the weight 2^-f, started from the
Chebyshev extrema. The fit is computed here in float64 and printed with the
fp32 values the kernel embeds. Run ``python exp2_poly_fit.py`` to reproduce.
"""
from __future__ import annotations

import numpy as np


def remez_relative(deg: int = 3, iters: int = 60, grid_points: int = 400001):
    """(coefficients c0..c_deg in float64, levelled relative error E)."""
    n = deg + 2
    k = np.arange(n)
    ref = 0.5 - 0.5 * np.cos(np.pi * k / (n - 1))          # Chebyshev extrema on [0, 1]
    grid = np.linspace(0.0, 1.0, grid_points)
    c, E = None, None
    for _ in range(iters):
        # p(x_i) - 2^x_i = (-1)^i * E * 2^x_i at the n reference points.
        A = np.zeros((n, n))
        A[:, :deg + 1] = ref[:, None] ** np.arange(deg + 1)[None, :]
        A[:, deg + 1] = -((-1.0) ** k) * np.exp2(ref)
        sol = np.linalg.solve(A, np.exp2(ref))
        c, E = sol[:deg + 1], sol[deg + 1]
        err = np.polynomial.polynomial.polyval(grid, c) / np.exp2(grid) - 1.0
        # One extremum per run of equal sign becomes the new reference.
        sign_change = np.nonzero(np.diff(np.sign(err)))[0] + 1
        bounds = np.concatenate(([0], sign_change, [grid.size]))
        ext = [lo + int(np.argmax(np.abs(err[lo:hi]))) for lo, hi in zip(bounds[:-1], bounds[1:])]
        if len(ext) > n:
            ext = sorted(sorted(ext, key=lambda j: -abs(err[j]))[:n])
        if len(ext) < n:
            break
        ref = grid[ext]
    return c, abs(E)


def coefficients_f32():
    c, _ = remez_relative()
    return [float(np.float32(x)) for x in c]


if __name__ == "__main__":
    c, E = remez_relative()
    print(f"levelled relative error: {E:.4e} (2^{np.log2(E):.2f})")
    for i, x in enumerate(c):
        f = np.float32(x)
        print(f"c{i} = {float(f)!r}f  (bits 0x{f.view(np.uint32):08x}, float64 {x!r})")

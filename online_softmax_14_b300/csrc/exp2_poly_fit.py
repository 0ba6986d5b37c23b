"""Fit the polynomial behind exp2_fma2() in exp2_poly.cuh.

    python online_softmax_14_b300/csrc/exp2_poly_fit.py     # prints the coefficients

The kernels evaluate 2^x for part of the softmax exponentials on the FMA pipe
instead of the special-function unit.  After Cody and Waite's range reduction
(W. J. Cody and W. Waite, "Software Manual for the Elementary Functions", 1980:
split x = n + f with n an integer, f = x - n, and rebuild 2^x = 2^n * 2^f), only
2^f for f in [-1/2, 1/2] needs a polynomial.  This script finds the degree-3
polynomial p minimising max |p(f) / 2^f - 1| on that interval with the Remez
exchange algorithm (E. Ya. Remez, 1934): solve for the coefficients and the
levelled error E on a reference of deg + 2 points, move the reference to the
extrema of the new error curve, repeat until the extrema are level.

The result, rounded to float32, is what exp2_poly.cuh holds; a CPU test re-runs
the fit and checks both the coefficients and the error bound.
"""

from __future__ import annotations

import mpmath as mp

DEGREE = 3
LO, HI = -0.5, 0.5


def remez_exp2(degree: int = DEGREE, lo: float = LO, hi: float = HI, iters: int = 40, grid: int = 4000):
    """Coefficients c_0..c_degree (float) of the minimax relative-error fit of
    2^f on [lo, hi], and the maximum relative error found on a dense grid."""
    mp.mp.dps = 40
    m = degree + 2
    # initial reference: Chebyshev extrema of the interval
    ref = [(lo + hi) / 2 - (hi - lo) / 2 * mp.cos(mp.pi * k / (m - 1)) for k in range(m)]
    coef = None
    for _ in range(iters):
        a = mp.matrix(m, m)
        rhs = mp.matrix(m, 1)
        for i, x in enumerate(ref):
            for k in range(degree + 1):
                a[i, k] = mp.mpf(x) ** k
            # p(x) - 2^x = (-1)^i E 2^x  (relative error levelled to +-E)
            a[i, degree + 1] = -((-1) ** i) * mp.power(2, x)
            rhs[i] = mp.power(2, x)
        sol = mp.lu_solve(a, rhs)
        coef = [sol[k] for k in range(degree + 1)]

        def rel_err(x):
            return sum(coef[k] * x ** k for k in range(degree + 1)) / mp.power(2, x) - 1

        xs = [lo + (hi - lo) * i / grid for i in range(grid + 1)]
        ev = [rel_err(mp.mpf(x)) for x in xs]
        # local extrema of |error|, then one per run of equal sign
        ext = [(xs[i], ev[i]) for i in range(len(xs))
               if i in (0, len(xs) - 1) or (abs(ev[i]) >= abs(ev[i - 1]) and abs(ev[i]) >= abs(ev[i + 1]))]
        runs = []
        for x, e in ext:
            if runs and mp.sign(runs[-1][1]) == mp.sign(e):
                if abs(e) > abs(runs[-1][1]):
                    runs[-1] = (x, e)
            else:
                runs.append((x, e))
        while len(runs) > m:  # drop the smaller end until the reference has m points
            runs = runs[1:] if abs(runs[0][1]) < abs(runs[-1][1]) else runs[:-1]
        ref = [x for x, _ in runs]
    return [float(c) for c in coef], float(max(abs(e) for e in ev))


if __name__ == "__main__":
    c, err = remez_exp2()
    for k, v in enumerate(c):
        print(f"c{k} = {v!r}  (float32 {float.hex(float(__import__('numpy').float32(v)))})")
    print(f"max relative error on [{LO}, {HI}]: {err:.3e}")

"""Fits the polynomial that device_math.cuh uses for log1p(e) on e in [0, 1].

log1p(e) = e * q(e) with q(e) = 1 + e * r(e); r is a degree-7 polynomial fitted
by iteratively reweighted least squares (Chebyshev basis, weights growing with
the relative error, so the result approaches a minimax fit of the relative
error of e * q(e)).  Prints the coefficients of r (lowest degree first) as
float32 and the maximum relative error of e * q(e) evaluated in float32 Horner
form against log1p in float64.

Usage: python fit_log1p.py
"""
import numpy as np
from numpy.polynomial import chebyshev as C


def fit(deg=7, rounds=6):
    e = np.linspace(1e-9, 1, 400001)
    r = (np.log1p(e) / e - 1) / e
    best, err = None, None
    for _ in range(rounds):
        w = None if err is None else np.abs(err) / np.abs(err).max() + 0.05
        coef = C.Chebyshev.fit(e, r, deg, domain=[0, 1], w=w).convert(kind=np.polynomial.Polynomial).coef
        coef = coef.astype(np.float32)
        x = e.astype(np.float32)
        acc = np.full_like(x, coef[-1])
        for c in coef[-2::-1]:
            acc = (acc * x + c).astype(np.float32)
        val = ((acc * x + np.float32(1)) * x).astype(np.float32).astype(np.float64)
        ref = np.log1p(x.astype(np.float64))
        err = (val - ref) / ref
        if best is None or np.abs(err).max() < best[0]:
            best = (float(np.abs(err).max()), coef)
    return best


if __name__ == "__main__":
    m, coef = fit()
    print("max relative error %.3e" % m)
    print(", ".join("%.9ef" % c for c in coef))

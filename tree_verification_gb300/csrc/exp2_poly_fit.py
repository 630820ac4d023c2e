"""Fits the polynomial 2^f ~ c0 + c1 f + c2 f^2 + c3 f^3 on [-1/2, 1/2] used by the
tree-attention kernel's FMA-pipe exponential (attention_tc.cu, exp2_poly2).

Relative-error least squares on Chebyshev nodes, refined by Lawson's iteration
toward the minimax solution; prints the float32 coefficients and the maximum
relative error of the float32 Horner evaluation.  Run: python exp2_poly_fit.py
"""
import numpy as np


def fit(deg=3, iters=200):
    f = np.cos(np.linspace(0.0, np.pi, 4001)) * 0.5
    y = np.exp2(f)
    A = np.vander(f, deg + 1, increasing=True) / y[:, None]
    b = np.ones_like(f)
    wt = np.ones_like(f)
    for _ in range(iters):
        sw = np.sqrt(wt)
        c = np.linalg.lstsq(A * sw[:, None], b * sw, rcond=None)[0]
        err = np.abs(A @ c - 1.0)
        wt = wt * (err / err.max() + 1e-12)
        wt /= wt.sum()
    c32 = c.astype(np.float32)
    x = np.linspace(-0.5, 0.5, 200001).astype(np.float32)
    p = np.full_like(x, c32[-1])
    for k in range(deg - 1, -1, -1):
        p = (p * x + c32[k]).astype(np.float32)
    return c32, float(np.abs(p.astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0).max())


if __name__ == "__main__":
    c, e = fit()
    print("coefficients:", ", ".join(f"{v:.9g}f" for v in c), " max relative error:", e)

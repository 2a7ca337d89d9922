"""Derives the coefficients of the polynomial exp2 used in the attention
softmax (attn_fwd_bf16.cu, ``exp2_poly``).

2^x is split as 2^n * 2^f with n = round(x) (obtained by adding and
subtracting 1.5 * 2^23, which leaves n in the low mantissa bits) and
f = x - n in [-1/2, 1/2].  2^f is approximated by a cubic p(f) chosen to
minimise the maximum RELATIVE error on [-1/2, 1/2] (Lawson's iteratively
reweighted least squares converges to the minimax solution), and n is added
to the exponent bits of p(f).  The probabilities that use it are rounded to bf16 (relative error
2^-9) right after, so a relative error near 1e-4 is invisible there.

Run: python exp2_poly_fit.py  -> prints the coefficients and the max error.
"""
import numpy as np


def fit(degree: int = 3, iters: int = 400):
    f = np.linspace(-0.5, 0.5, 20001)
    y = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True)
    w = np.ones_like(f)
    for _ in range(iters):
        sw = np.sqrt(w) / y                       # relative error weighting
        c, *_ = np.linalg.lstsq(V * sw[:, None], y * sw, rcond=None)
        err = np.abs(V @ c - y) / y
        w = w * err
        w /= w.sum()
    err = (V @ c - y) / y
    return c, float(np.abs(err).max())


if __name__ == "__main__":
    c, e = fit()
    print("coefficients c0..c3:", ", ".join(f"{x:.9g}f" for x in c))
    print("max relative error on [-1/2, 1/2]:", e)

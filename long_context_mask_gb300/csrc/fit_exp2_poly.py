"""Fit the polynomial used by the kernel's FMA-pipe exp2.

Method (Cody and Waite range reduction, polynomial by a minimax fit):
    2^x = 2^j * 2^f,   j = round(x),  f = x - j in [-1/2, 1/2]
and 2^f is approximated by a degree-3 polynomial p(f) whose coefficients
minimise the maximum RELATIVE error |p(f) / 2^f - 1| over [-1/2, 1/2].  The
minimax solution is found by Lawson's iteratively reweighted least squares
on a dense grid (weights multiplied by the current error each round), which
converges to the equioscillating (Chebyshev) solution.  The constant term is
left free; its small offset from 1 halves the peak error.

Run: python fit_exp2_poly.py   -> prints the coefficients as C hex floats and
the achieved relative error in float64 and in float32 Horner evaluation.
The softmax rounds p to bf16 (relative step 2^-8), so any relative error well
below 2^-9 ~ 2e-3 is invisible in the output.
"""
import numpy as np

DEGREE = 3


def fit(degree=DEGREE, n=20001, rounds=200):
    f = np.linspace(-0.5, 0.5, n)
    y = np.exp2(f)
    A = np.vander(f, degree + 1, increasing=True) / y[:, None]  # relative error rows
    b = np.ones_like(f)
    w = np.ones_like(f) / n
    c = None
    for _ in range(rounds):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], b * sw, rcond=None)
        err = np.abs(A @ c - b)
        w = w * err
        w /= w.sum()
    return c


def rel_error_f32(c, n=1 << 20):
    f = np.linspace(-0.5, 0.5, n, dtype=np.float32)
    c32 = c.astype(np.float32)
    p = np.full_like(f, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        p = (p * f + c32[k]).astype(np.float32)
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1)))


if __name__ == "__main__":
    c = fit()
    f = np.linspace(-0.5, 0.5, 100001)
    e64 = np.max(np.abs(np.polyval(c[::-1], f) / np.exp2(f) - 1))
    for k, ck in enumerate(c):
        print(f"c{k} = {float(np.float32(ck)).hex()}f  // {np.float32(ck)!r}")
    print(f"max relative error: {e64:.3e} (fp64), {rel_error_f32(c):.3e} (fp32 Horner)")

"""Fits the polynomial of the software exp2 in exp2_poly.cuh.

2^x = 2^n * 2^f with n = x rounded to the nearest integer and f = x - n in
[-1/2, 1/2] (Cody and Waite's range reduction: the exponent takes n, a
polynomial takes 2^f).  Here 2^f ~ 1 + f*(c1 + f*(c2 + f*c3)): the constant
term is pinned to 1 so that an integer x gives an exact power of two.  The
coefficients minimise the largest relative error over [-1/2, 1/2]: Lawson's
iteration (a least-squares fit whose weights grow where the error is
largest) converges to the minimax fit.  They are then rounded to float32 and
the error is measured again with the polynomial evaluated in float32 (fused
multiply-adds, as on the GPU).

    python fit_exp2_poly.py        prints the float32 coefficients (hex and
                                   decimal) and the measured error
"""
import numpy as np

DEGREE = 3
LAWSON_ITERS = 400


def fit(degree=DEGREE, iters=LAWSON_ITERS, n_nodes=4001):
    f = np.cos(np.linspace(0.0, np.pi, n_nodes)) * 0.5  # Chebyshev-spaced points of [-1/2, 1/2]
    target = np.exp2(f)
    # unknowns c1..c_degree of 1 + sum_k c_k f^k; relative error (p - t) / t
    A = np.stack([f ** k for k in range(1, degree + 1)], axis=1) / target[:, None]
    b = (target - 1.0) / target
    w = np.full(n_nodes, 1.0 / n_nodes)
    c = None
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], b * sw, rcond=None)
        err = np.abs(A @ c - b)
        w = w * err
        w /= w.sum()
    return c


def eval_f32(c32, f):
    """1 + f*(c1 + f*(c2 + f*c3)) in float32 with fused multiply-adds."""
    f = np.asarray(f, dtype=np.float32).astype(np.float64)
    p = np.float64(c32[-1])
    for ck in c32[-2::-1]:
        p = np.float32(p * f + np.float64(ck)).astype(np.float64)  # fma: one rounding
    return np.float32(p * f + 1.0).astype(np.float64)


def rel_error_f32(c32, n=200001):
    f = np.linspace(-0.5, 0.5, n).astype(np.float32)
    return float(np.max(np.abs(eval_f32(c32, f) / np.exp2(f.astype(np.float64)) - 1.0)))


def coefficients():
    c = fit()
    return [np.float32(x) for x in c]


if __name__ == "__main__":
    c32 = coefficients()
    for k, x in enumerate(c32, start=1):
        print("c%d = %.9ef  (0x%08x)" % (k, float(x), np.array(x, dtype=np.float32).view(np.uint32)))
    print("max relative error over [-1/2, 1/2], float32 evaluation: %.3e" % rel_error_f32(c32))

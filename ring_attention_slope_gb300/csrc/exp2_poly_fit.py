"""Fits the cubic used by the attention kernel's FMA-pipe exp2 (softmax_pair_poly).

2^x is split as 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]
(Cody-Waite range reduction; the rounding is done by adding 1.5 * 2^23).  On
that interval 2^f is approximated by 1 + c1 f + c2 f^2 + c3 f^3.  The constant
term is held at exactly 1 so that every integer x (in particular x = 0, the row
maximum of a softmax) gives its power of two exactly.  c1..c3 are fitted for the
smallest maximum RELATIVE error with Lawson's iteratively reweighted least
squares on Chebyshev nodes (the weights converge to the minimax solution).  The
coefficients are then rounded to float32 and the error of the float32 Horner
evaluation is measured on a dense grid.

Run: python exp2_poly_fit.py  (prints the coefficients as float32 hex literals
for sm103_ptx.cuh and the measured maximum relative error).
"""
import numpy as np

DEGREE = 3


def fit(degree=DEGREE, nodes=4001, iters=400):
    """Returns [1, c1, ..., c_degree] (float64)."""
    k = np.arange(nodes)
    f = 0.5 * np.cos(np.pi * (k + 0.5) / nodes)  # Chebyshev nodes on [-1/2, 1/2]
    y = np.exp2(f)
    # relative error (1 + sum c_i f^i) / y - 1 = rows @ c - target
    rows = np.stack([f**i for i in range(1, degree + 1)], axis=1) / y[:, None]
    target = (y - 1.0) / y
    w = np.full(nodes, 1.0 / nodes)
    coef = None
    for _ in range(iters):
        sw = np.sqrt(w)
        coef, *_ = np.linalg.lstsq(rows * sw[:, None], target * sw, rcond=None)
        err = np.abs(rows @ coef - target)
        w = w * err
        w /= w.sum()
    return np.concatenate([[1.0], coef])


def horner_f32(coef32, f):
    """Float32 Horner evaluation with one rounding per fused multiply-add, as the kernel does it."""
    f = f.astype(np.float32)
    q = np.full_like(f, coef32[-1])
    for c in coef32[-2::-1]:
        q = (q.astype(np.float64) * f.astype(np.float64) + np.float64(c)).astype(np.float32)
    return q


def max_rel_error(coef32):
    f = np.linspace(-0.5, 0.5, 2_000_001, dtype=np.float64).astype(np.float32)
    return float(np.max(np.abs(horner_f32(coef32, f).astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)))


def hex_f32(v):
    return "0f%08X" % np.float32(v).view(np.uint32)


if __name__ == "__main__":
    c = fit()
    c32 = c.astype(np.float32)
    for i, v in enumerate(c32):
        print(f"c{i} = {float(v)!r:24} {hex_f32(v)}")
    print(f"max relative error of the float32 evaluation on [-1/2, 1/2]: {max_rel_error(c32):.3e}")

"""Derives the polynomial that the kernels use to evaluate 2^x on the FMA pipe.

2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2].  2^f is
approximated by the degree-3 polynomial p(f) = c0 + c1 f + c2 f^2 + c3 f^3
that minimises the maximum RELATIVE error max |p(f) / 2^f - 1| over
[-1/2, 1/2], found with the Remez exchange algorithm (equioscillation at
five points).  2^n is applied by adding n to the exponent field.

Run:  python gen_exp2_poly.py   -> prints the coefficients (as float32 hex
and decimal) and the error bound.  The same constants appear in
sm103_ptx.cuh (exp2_fma); tests/test_exp2_poly.py checks that they agree
with this derivation and that the float32 evaluation meets the bound.
"""
import numpy as np


def remez_exp2(deg: int = 3, lo: float = -0.5, hi: float = 0.5, iters: int = 30):
    # initial reference: Chebyshev extrema mapped to [lo, hi]
    m = deg + 2
    k = np.arange(m)
    x = (lo + hi) / 2 + (hi - lo) / 2 * np.cos(np.pi * (m - 1 - k) / (m - 1))
    grid = np.linspace(lo, hi, 200001)
    c = None
    E = 0.0
    for _ in range(iters):
        # solve p(x_i) - 2^x_i = (-1)^i E 2^x_i for c0..c_deg and E
        A = np.zeros((m, m))
        for i in range(m):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2.0 ** x[i]
        sol = np.linalg.solve(A, 2.0 ** x)
        c, E = sol[:deg + 1], sol[deg + 1]
        err = np.polyval(c[::-1], grid) / 2.0 ** grid - 1.0
        # new reference: one extremum of err per sign-alternating segment
        sign = np.sign(err)
        idx = np.where(np.diff(sign) != 0)[0]
        bounds = np.concatenate([[0], idx + 1, [len(grid)]])
        ext = [b0 + int(np.argmax(np.abs(err[b0:b1]))) for b0, b1 in zip(bounds[:-1], bounds[1:])]
        if len(ext) != m:
            break
        x = grid[ext]
    err = np.polyval(c[::-1], grid) / 2.0 ** grid - 1.0
    return c, float(np.max(np.abs(err)))


def coefficients_f32():
    c, bound = remez_exp2()
    return [float(np.float32(v)) for v in c], bound


if __name__ == "__main__":
    cf, bound = coefficients_f32()
    for i, v in enumerate(cf):
        print(f"c{i} = {v:.9e}f  (0x{np.float32(v).view(np.uint32):08x})")
    print(f"max relative error of p(f) vs 2^f on [-1/2, 1/2]: {bound:.3e}")

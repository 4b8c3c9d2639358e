"""Derives the polynomial used by the kernels' FMA-pipe exp2.

2^x is split Cody-Waite style into 2^n * 2^f with n = round(x) and
f = x - n in [-1/2, 1/2]; 2^f is approximated by a degree-4 polynomial whose
coefficients minimise the maximum relative error on [-1/2, 1/2] (a few Remez
exchange steps started from a Chebyshev-node least-squares fit).  Running this
file prints the coefficients as float32 literals and the error bound; the
kernels carry the printed values.
"""
import numpy as np

DEG = 4
LO, HI = -0.5, 0.5


def fit(deg=DEG, iters=30):
    # Remez on the relative error e(f) = p(f) / 2^f - 1
    k = np.arange(deg + 2)
    xs = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * (deg + 1 - k) / (deg + 1))
    grid = np.linspace(LO, HI, 200001)
    c = None
    for _ in range(iters):
        # solve p(x_i) / 2^x_i - 1 = (-1)^i E  for c_0..c_deg, E
        A = np.zeros((deg + 2, deg + 2))
        for i, x in enumerate(xs):
            A[i, :deg + 1] = x ** np.arange(deg + 1) / 2.0 ** x
            A[i, deg + 1] = -((-1) ** i)
        sol = np.linalg.solve(A, np.ones(deg + 2))
        c = sol[:deg + 1]
        err = np.polyval(c[::-1], grid) / 2.0 ** grid - 1
        # new reference: extrema of the error, one per sign change segment
        idx = [0]
        for j in range(1, len(grid) - 1):
            if (err[j] - err[j - 1]) * (err[j + 1] - err[j]) < 0:
                idx.append(j)
        idx.append(len(grid) - 1)
        if len(idx) != deg + 2:
            break
        xs = grid[idx]
    return c


def eval_f32(c32, x):
    """The kernel's arithmetic, in float32: round-to-nearest split through the
    1.5 * 2^23 shifter, Horner in f32, exponent added to the bit pattern."""
    x = np.maximum(x.astype(np.float32), np.float32(-127.0))
    sh = np.float32(12582912.0)
    t = (x + sh).astype(np.float32)
    n = (t - sh).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.float32(c32[DEG])
    for i in range(DEG - 1, -1, -1):
        p = (p * f + np.float32(c32[i])).astype(np.float32)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return bits.astype(np.int32).view(np.float32)


if __name__ == "__main__":
    c = fit()
    c32 = c.astype(np.float32)
    xs = np.linspace(-30, 8, 2_000_001).astype(np.float32)
    rel = np.abs(eval_f32(c32, xs).astype(np.float64) / np.exp2(xs.astype(np.float64)) - 1)
    for i, v in enumerate(c32):
        print(f"c{i} = {float(v).hex()}  ({float(v):.9e})")
    print(f"max relative error of the f32 evaluation on [-30, 8]: {rel.max():.3e}")

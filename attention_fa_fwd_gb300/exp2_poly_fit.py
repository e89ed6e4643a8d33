"""Fit of the polynomial behind the FMA-pipe exponential `ptx::f2_exp2_poly`.

The softmax computes p = 2^x.  On the FMA pipe 2^x is split as 2^n * 2^f with
n = rint(x) and f = x - n in [-1/2, 1/2]; 2^n goes straight into the exponent
field and 2^f comes from a polynomial.  P is rounded to fp16 or bf16 (11 or 8
significand bits) right after, so a relative error well under 2^-12 is enough:
degree 3 reaches 7.5e-5.

The coefficients minimise the maximum *relative* error on [-1/2, 1/2] (a
Remez exchange with weight 1/2^f: solve for the polynomial that equioscillates
on deg + 2 reference points, move the points to the extrema of the error,
repeat).  Running this file prints them as fp32 literals, the form they take
in the CUDA source, and the error of the fp32 Horner evaluation.

    python attention_fa_fwd_gb300/exp2_poly_fit.py
"""
import numpy as np

LO, HI = -0.5, 0.5


def remez_relative(deg, iters=40, grid=200001):
    n = deg + 2
    # start from Chebyshev extrema
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    g = np.linspace(LO, HI, grid)
    for _ in range(iters):
        a = np.zeros((n, n))
        for i in range(n):
            a[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            a[i, deg + 1] = (-1) ** i * np.exp2(x[i])   # relative error: E * 2^x
        sol = np.linalg.solve(a, np.exp2(x))
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], g) - np.exp2(g)) / np.exp2(g)
        # local extrema of the error (and the interval ends), one per sign run
        turns = np.nonzero((err[1:-1] - err[:-2]) * (err[2:] - err[1:-1]) <= 0)[0] + 1
        ext = [0] + turns.tolist() + [grid - 1]
        sel = []
        for i in ext:
            if sel and np.sign(err[i]) == np.sign(err[sel[-1]]):
                if abs(err[i]) > abs(err[sel[-1]]):
                    sel[-1] = i
            else:
                sel.append(i)
        while len(sel) > n:
            sel.pop(0 if abs(err[sel[0]]) < abs(err[sel[-1]]) else -1)
        if len(sel) == n:
            x = g[sel]
    return c, float(np.max(np.abs(err)))


def horner_f32(c32, f):
    p = np.float32(c32[-1])
    for ck in c32[-2::-1]:
        p = (p * f + ck).astype(np.float32)
    return p


def fp32_error(c32):
    f = np.linspace(LO, HI, 1000001).astype(np.float32)
    p = horner_f32(c32, f).astype(np.float64)
    ref = np.exp2(f.astype(np.float64))
    return float(np.max(np.abs(p - ref) / ref))


if __name__ == "__main__":
    for deg in (2, 3, 4):
        c, e = remez_relative(deg)
        c32 = c.astype(np.float32)
        print(f"degree {deg}: max relative error {e:.3e} (fp32 Horner {fp32_error(c32):.3e})")
        print("    c0..c%d = %s" % (deg, ", ".join(f"{float(v):.10g}f" for v in c32)))

"""Coefficients of the FMA-pipe base-2 exponential used by the score kernels.

Method (Cody & Waite range reduction, then a minimax polynomial): write
x = j + f with j = rint(x) and f in [-1/2, 1/2]; 2^x = 2^j * p(f).  p is the
polynomial of the given degree that minimises max |p(f) / 2^f - 1| on
[-1/2, 1/2], found with the Remez exchange algorithm (solve for equal
alternating relative error on n+2 reference points, move the references to
the extrema of the error, repeat).  2^j is applied by adding j to the
float's exponent field.

Run this file to print the fp32 coefficients and their maximum relative
error; the kernel embeds the printed values.
"""
import numpy as np


def remez(deg, iters=30, grid=200001, lo=-0.5, hi=0.5):
    n = deg + 2
    # Chebyshev extrema as the first reference set
    k = np.arange(n)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * k[::-1] / (n - 1))
    fine = np.linspace(lo, hi, grid)
    for _ in range(iters):
        t = np.exp2(x)
        # p(x_i) - (-1)^i E t_i = t_i
        A = np.hstack([np.vander(x, deg + 1, increasing=True),
                       (-(-1.0) ** np.arange(n) * t)[:, None]])
        sol = np.linalg.solve(A, t)
        c = sol[:-1]
        err = np.polyval(c[::-1], fine) / np.exp2(fine) - 1.0
        # new references: the extremum of each run of constant error sign
        sgn = np.sign(err)
        idx, start = [], 0
        for i in range(1, grid + 1):
            if i == grid or sgn[i] != sgn[start]:
                seg = np.arange(start, i)
                idx.append(seg[np.argmax(np.abs(err[seg]))])
                start = i
        if len(idx) < n:
            break
        if len(idx) > n:   # keep the n largest alternating extrema
            while len(idx) > n:
                e = np.abs(err[idx])
                drop = 0 if e[0] < e[-1] else len(idx) - 1
                idx.pop(drop)
        x = fine[np.array(idx)]
    return c


def max_rel_err(c32, n=400001):
    f = np.linspace(-0.5, 0.5, n, dtype=np.float64)
    p = np.zeros_like(f)
    for ck in np.asarray(c32, dtype=np.float64)[::-1]:
        p = p * f + ck
    return float(np.max(np.abs(p / np.exp2(f) - 1.0)))


if __name__ == "__main__":
    import sys
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 4
    c = remez(deg).astype(np.float32)
    for i, ck in enumerate(c):
        print(f"C{i} = {float(ck)!r}f  // {np.float32(ck).view(np.uint32):#010x}")
    print("max relative error of the fp32 coefficients:", max_rel_err(c))

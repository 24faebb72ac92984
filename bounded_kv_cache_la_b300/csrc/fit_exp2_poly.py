"""Fits the polynomial the tensor-core attention uses for part of its
exponentials (2^f on f in [-1/2, 1/2], minimax in relative error).

Method: Remez exchange on the relative error e(f) = p(f) / 2^f - 1 for a
polynomial of degree 3, then rounding of the coefficients to fp32 and a
dense check of the error with fp32 Horner evaluation.  The kernel forms
2^x = 2^n * 2^f with n = rint(x) (Cody and Waite's argument reduction,
which is exact here because the base is 2).

Run: python bounded_kv_cache_la_b300/csrc/fit_exp2_poly.py
"""
import numpy as np

DEG = 3
LO, HI = -0.5, 0.5


def remez(deg=DEG, iters=30):
    n = deg + 2
    # Chebyshev extrema as the first reference
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    dense = np.linspace(LO, HI, 200001)
    for _ in range(iters):
        # p(x_i) - 2^x_i = (-1)^i E 2^x_i  (relative equioscillation)
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2.0 ** x[i]
        sol = np.linalg.solve(A, 2.0 ** x)
        c = sol[:deg + 1]
        err = np.polyval(c[::-1], dense) / 2.0 ** dense - 1.0
        # new reference: extrema of err between sign changes
        idx = [0]
        for k in range(1, len(dense) - 1):
            if (err[k] - err[k - 1]) * (err[k + 1] - err[k]) <= 0 and abs(err[k]) > 1e-300:
                idx.append(k)
        idx.append(len(dense) - 1)
        idx = np.array(sorted(set(idx)))
        cand = dense[idx]
        if len(cand) >= n:
            # keep the n points with alternating signs and largest |err|
            sel = [idx[0]]
            for k in idx[1:]:
                if np.sign(err[k]) == np.sign(err[sel[-1]]):
                    if abs(err[k]) > abs(err[sel[-1]]):
                        sel[-1] = k
                else:
                    sel.append(k)
            if len(sel) >= n:
                sel = sorted(sel, key=lambda k: -abs(err[k]))[:n]
                x = np.sort(dense[sel])
    return c


def check(c32):
    f = np.linspace(LO, HI, 2000001).astype(np.float32)
    p = np.float32(c32[3])
    for k in (2, 1, 0):
        p = (p * f + np.float32(c32[k])).astype(np.float32)
    rel = p.astype(np.float64) / 2.0 ** f.astype(np.float64) - 1.0
    return float(np.max(np.abs(rel)))


if __name__ == "__main__":
    c = remez()
    c32 = [np.float32(v) for v in c]
    print("coefficients (c0 + c1 f + c2 f^2 + c3 f^3):")
    for k, v in enumerate(c32):
        print(f"  c{k} = {float(v)!r:>24}  ({v.view(np.uint32):#010x})")
    print(f"max relative error with fp32 Horner on [-1/2, 1/2]: {check(c32):.3e}")

"""Coefficients of the polynomial exp2 used for part of the softmax exponentials.

Method (Cody & Waite range reduction; Remez exchange for the minimax fit):
  x = n + f with n = round(x) (integer), f in [-1/2, 1/2];
  2^x = 2^n * p(f),  p(f) = c0 + c1 f + c2 f^2 + c3 f^3,
where c0..c3 minimise max |p(f) / 2^f - 1| on [-1/2, 1/2] (relative error).
2^n is applied by adding n to the IEEE exponent field.  The degree is chosen
for bf16 probabilities (8-bit mantissa): the fit's relative error is ~1e-4.

Run `python -m persistent_sm_ring_gb300.exp2_poly` to print the coefficients
as C hex floats (they are pasted into csrc/psr_device.cuh) and the error.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def _error(c, f):
    p = sum(ck * f ** k for k, ck in enumerate(c))
    return p / np.exp2(f) - 1.0


def remez(degree: int = DEGREE, iters: int = 60):
    """Minimax relative-error fit of 2^f by sum_{k=0..degree} c_k f^k on [LO, HI]."""
    n = degree + 2  # reference points: unknowns c_0..c_degree and the levelled error E
    # Chebyshev-like initial reference
    ref = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    grid = np.linspace(LO, HI, 200001)
    c = np.zeros(degree + 1)
    for _ in range(iters):
        # p(f_i) - 2^f_i = (-1)^i E 2^f_i  ->  sum_k c_k f_i^k - (-1)^i E 2^f_i = 2^f_i
        A = np.zeros((n, n))
        b = np.exp2(ref)
        for i, f in enumerate(ref):
            A[i, :degree + 1] = [f ** k for k in range(degree + 1)]
            A[i, degree + 1] = -((-1) ** i) * np.exp2(f)
        sol = np.linalg.solve(A, b)
        c = sol[:degree + 1]
        e = _error(c, grid)
        # new reference: the extremum of each sign-alternating run of the error curve
        sign = np.sign(e)
        idx = []
        start = 0
        for j in range(1, len(grid) + 1):
            if j == len(grid) or sign[j] != sign[start]:
                seg = slice(start, j)
                idx.append(start + int(np.argmax(np.abs(e[seg]))))
                start = j
        if len(idx) >= n:
            # keep n alternating points with the largest errors, in order
            while len(idx) > n:
                drop = int(np.argmin(np.abs(e[idx])))
                if drop in (0, len(idx) - 1):
                    idx.pop(drop)
                else:
                    idx.pop(drop)
            ref = grid[idx]
    return c, float(np.max(np.abs(_error(c, grid))))


def f32_emulate(c32, x):
    """The device sequence in float32: t = x + 1.5*2^23; n = t - 1.5*2^23; f = x - n;
    p = ((c3 f + c2) f + c1) f + c0 (fused multiply-adds); result bits = bits(p) + (n << 23)."""
    x = np.asarray(x, dtype=np.float32)
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    nn = (t - magic).astype(np.float32)
    f = (x - nn).astype(np.float32)

    c0, c1, c2, c3 = (np.float32(v) for v in c32)
    p = (f.astype(np.float64) * np.float64(c3) + np.float64(c2)).astype(np.float32)
    p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(c1)).astype(np.float32)
    p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(c0)).astype(np.float32)
    bits = p.view(np.int32) + (nn.astype(np.int32) << 23)
    return bits.view(np.float32)


def main():
    c, err = remez()
    c32 = [float(np.float32(v)) for v in c]
    x = np.linspace(-125.0, 8.0, 2_000_001).astype(np.float32)
    rel = np.abs(f32_emulate(c32, x).astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)
    print("minimax relative error (real arithmetic): %.3e" % err)
    print("float32 device sequence, max relative error on [-125, 8]: %.3e" % rel.max())
    for k, v in enumerate(c32):
        print("c%d = %s  (%.9g)" % (k, float(v).hex(), v))


if __name__ == "__main__":
    main()

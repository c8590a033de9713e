"""Fit of the cubic that the flash-attention softmax uses for part of its exponentials.

The softmax of the prefill attention kernel evaluates one exp2 per visible (query, key)
pair.  The multi-function unit (ex2.approx) that does this is the bottleneck of the softmax
warps, so a share of the exponentials is computed on the FMA pipe instead (flash_prefill.cuh,
exp2_fma2 in ptx.cuh), in the usual two steps:

  range reduction  a = j + f with j = rint(a) (round half to even), f in [-1/2, 1/2]:
                   t = a + 1.5 * 2^23 in fp32 leaves j in the low mantissa bits of t, and
                   j = t - 1.5 * 2^23, f = a - j are exact (Cody and Waite's additive
                   reduction, with the fp32 addition doing the rounding);
  approximation    2^f ~ p(f) = c0 + f (c1 + f (c2 + f c3)), Horner with fma;
  reconstruction   2^a ~ p(f) * 2^j by adding j to p's exponent field: bits(p) + (bits(t) << 23)
                   (the shift keeps the 9 low bits of t, i.e. j mod 512, in the exponent field).

The input is clamped to a >= -125 first, so that j >= -125 keeps the result a normal number.

The coefficients minimise the maximum RELATIVE error |p(f) / 2^f - 1| over [-1/2, 1/2]: a
Remez exchange (solve p(x_i) - 2^x_i = (-1)^i E 2^x_i on 5 reference points, move the points
to the extrema of the error curve, repeat until the levelled error E stops changing), then the
coefficients are rounded to fp32.  The error of the fp32 evaluation is measured by emulating
the device sequence step by step in numpy (fp32 adds; each fma as one fp32 rounding of the
exact product-sum).  P is stored in bf16 after the exponential (relative rounding error up to
2^-9), so the cubic's ~7.5e-5 adds little; a quadratic (~1.7e-3) would not.

Run as a script to print the coefficients (as fp32 hex) and the bounds.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5
ROUND = np.float32(12582912.0)  # 1.5 * 2^23
CLAMP = np.float32(-125.0)


def remez_relative(degree: int = DEGREE, lo: float = LO, hi: float = HI, iters: int = 40, grid_n: int = 200001):
    """Minimax coefficients (c0..c_degree, fp64) of p(x) ~ 2^x on [lo, hi] in relative error,
    and the levelled error E."""
    n = degree + 2
    k = np.arange(n)
    x = (lo + hi) / 2 + (hi - lo) / 2 * np.cos(np.pi * (n - 1 - k) / (n - 1))  # Chebyshev extrema
    grid = np.linspace(lo, hi, grid_n)
    E_prev = None
    for _ in range(iters):
        g = np.exp2(x)
        A = np.empty((n, n))
        for j in range(degree + 1):
            A[:, j] = x ** j
        A[:, degree + 1] = (-1.0) ** k * g
        sol = np.linalg.solve(A, g)
        c, E = sol[:degree + 1], sol[degree + 1]
        err = np.polyval(c[::-1], grid) / np.exp2(grid) - 1.0
        # one extremum per run of constant sign, then the n consecutive ones with the largest minimum
        sign = np.sign(err)
        ext, start = [], 0
        for i in range(1, grid_n):
            if sign[i] != sign[start]:
                ext.append(start + int(np.argmax(np.abs(err[start:i]))))
                start = i
        ext.append(start + int(np.argmax(np.abs(err[start:]))))
        if len(ext) > n:
            s0 = max(range(len(ext) - n + 1), key=lambda s: np.min(np.abs(err[ext[s:s + n]])))
            ext = ext[s0:s0 + n]
        x = grid[np.array(ext)]
        if E_prev is not None and abs(abs(E) - abs(E_prev)) <= 1e-12 * abs(E):
            break
        E_prev = E
    return c, abs(E)


def coefficients_f32():
    c, _ = remez_relative()
    return c.astype(np.float32)


def _fma32(a, b, c):
    # one fp32 rounding of a*b + c (the product of two fp32 values is exact in fp64)
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def exp2_emulated(a, coeffs=None) -> np.ndarray:
    """The device sequence of exp2_fma2 on fp32 inputs, step for step, in numpy."""
    c = coefficients_f32() if coeffs is None else np.asarray(coeffs, dtype=np.float32)
    a = np.maximum(np.asarray(a, dtype=np.float32), CLAMP)
    t = (a + ROUND).astype(np.float32)
    j = (t - ROUND).astype(np.float32)
    f = (a - j).astype(np.float32)
    p = np.full_like(f, c[3])
    for ck in (c[2], c[1], c[0]):
        p = _fma32(p, f, np.full_like(f, ck))
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(np.float32)


def main():
    c64, E = remez_relative()
    c = c64.astype(np.float32)
    print(f"levelled relative error of the minimax cubic: {E:.3e}")
    for i, v in enumerate(c):
        print(f"c{i} = {float(v).hex()}f  // {float(v):.9g}")
    a = np.linspace(-125.0, 8.0, 2_000_001, dtype=np.float32)
    rel = np.abs(exp2_emulated(a, c).astype(np.float64) / np.exp2(a.astype(np.float64)) - 1)
    print(f"fp32 evaluation, a in [-125, 8]: max relative error {rel.max():.3e}")


if __name__ == "__main__":
    main()

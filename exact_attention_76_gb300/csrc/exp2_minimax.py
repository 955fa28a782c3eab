"""Coefficients of the polynomial exp2 used by the forward kernel's softmax.

Part of the exponentials of the softmax are evaluated on the FMA pipes instead
of the special-function unit ("software exp2" of FlashAttention-4 in
"FlashAttention 源码级深度解析", timeline and summary).  The method is:

* range reduction after Cody and Waite (W. J. Cody, W. Waite, "Software Manual
  for the Elementary Functions", 1980): ``x = n + f`` with ``n = round(x)``, so
  ``2^x = 2^n * 2^f`` and ``f`` lies in ``[-1/2, 1/2]``; ``2^n`` is applied by
  adding ``n`` to the exponent field of ``2^f``;
* ``2^f`` on ``[-1/2, 1/2]`` by the polynomial of the given degree that
  minimises the largest RELATIVE error, found with the Remez exchange algorithm
  (E. Remez, 1934) in float64 and then rounded to float32.

Run ``python exp2_minimax.py`` to print the coefficients; the kernel carries
them as literals and a CPU test checks the two agree and bounds the error of
the float32 evaluation.
"""
from __future__ import annotations

import numpy as np

LO, HI = -0.5, 0.5


def _fit_on_reference(xs: np.ndarray, degree: int) -> tuple[np.ndarray, float]:
    """Solves p(x_i) - 2^x_i = (-1)^i E 2^x_i for the coefficients and E."""
    k = degree + 2
    a = np.zeros((k, k))
    for i, x in enumerate(xs):
        a[i, : degree + 1] = x ** np.arange(degree + 1)
        a[i, degree + 1] = -((-1) ** i) * 2.0**x
    sol = np.linalg.solve(a, 2.0**xs)
    return sol[: degree + 1], float(sol[degree + 1])


def _rel_err(c: np.ndarray, x: np.ndarray) -> np.ndarray:
    return np.polynomial.polynomial.polyval(x, c) / 2.0**x - 1.0


def remez(degree: int, iters: int = 30, grid: int = 200001) -> tuple[np.ndarray, float]:
    """Minimax (relative error) polynomial for 2^f on [LO, HI]; returns
    (coefficients c_0..c_degree in float64, max relative error)."""
    k = degree + 2
    # Chebyshev extrema as the first reference
    xs = 0.5 * (LO + HI) - 0.5 * (HI - LO) * np.cos(np.pi * np.arange(k) / (k - 1))
    fine = np.linspace(LO, HI, grid)
    c = None
    for _ in range(iters):
        c, _ = _fit_on_reference(xs, degree)
        e = _rel_err(c, fine)
        # new reference: one extremum of |e| per run of constant sign
        sign = np.sign(e)
        sign[sign == 0] = 1
        cuts = np.flatnonzero(np.diff(sign)) + 1
        runs = np.split(np.arange(grid), cuts)
        ext = np.array([r[np.argmax(np.abs(e[r]))] for r in runs])
        if len(ext) > k:  # keep the k largest consecutive alternating extrema
            best, best_val = 0, -1.0
            for s in range(len(ext) - k + 1):
                v = np.min(np.abs(e[ext[s : s + k]]))
                if v > best_val:
                    best, best_val = s, v
            ext = ext[best : best + k]
        if len(ext) < k:
            break
        xs = fine[ext]
    return c, float(np.max(np.abs(_rel_err(c, fine))))


def coefficients_f32(degree: int) -> np.ndarray:
    """The coefficients c_0..c_degree rounded to float32."""
    c, _ = remez(degree)
    return c.astype(np.float32)


def _fma32(a, b, c):
    # float32 fused multiply-add: the product of two float32 is exact in float64
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def eval_exp2_f32(x: np.ndarray, c32: np.ndarray, clamp: float = -126.0) -> np.ndarray:
    """The kernel's evaluation, step for step in float32: clamp, round to the
    nearest integer with the 1.5 * 2^23 shifter, Horner with FMAs, and the
    integer add of n into the exponent field."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(clamp))
    shifter = np.float32(12582912.0)
    t = (x + shifter).astype(np.float32)
    nf = (t - shifter).astype(np.float32)
    f = (x - nf).astype(np.float32)
    p = np.full_like(f, c32[-1])
    for ci in c32[-2::-1]:
        p = _fma32(p, f, np.full_like(f, ci))
    bits = p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << np.uint64(23))
    return (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)


def main() -> None:
    for degree in (2, 3):
        c, err = remez(degree)
        c32 = c.astype(np.float32)
        print(f"degree {degree}: max relative error {err:.3e} (float64 coefficients)")
        print("  float32:", ", ".join(f"{float(v):.9g}f" for v in c32))


if __name__ == "__main__":
    main()

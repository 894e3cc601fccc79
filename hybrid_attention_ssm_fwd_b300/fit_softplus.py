"""Fits the polynomial behind the scan kernel's softplus.

    python -m hybrid_attention_ssm_fwd_b300.fit_softplus

softplus(v) = max(v, 0) + log1p(e) with e = exp(-|v|) in (0, 1].  The kernel
evaluates log1p(e) as e * q(e), q a degree-7 polynomial approximating
f(e) = log1p(e) / e on [0, 1] (f(0) = 1), so that a single exponential and
seven FMAs give softplus with no branch and no logarithm.

The fit is Lawson's iteratively reweighted least squares for the minimax
(equal-ripple) relative error: start from a least-squares fit on Chebyshev
nodes of [0, 1], then multiply each node's weight by its current absolute
relative error and refit, which drives the weighted solution toward the
minimax one.  Coefficients are returned highest degree first (the Horner
order the kernel uses) and rounded to float32.
"""
from __future__ import annotations

import numpy as np

DEGREE = 7


def target(e: np.ndarray) -> np.ndarray:
    """log1p(e) / e, with its limit 1 at e = 0."""
    e = np.asarray(e, np.float64)
    out = np.ones_like(e)
    nz = e > 0
    out[nz] = np.log1p(e[nz]) / e[nz]
    return out


def fit(degree: int = DEGREE, nodes: int = 400, iters: int = 60) -> np.ndarray:
    """Minimax-relative-error polynomial coefficients of target() on [0, 1],
    highest degree first, rounded to float32."""
    k = np.arange(nodes)
    x = 0.5 - 0.5 * np.cos((2 * k + 1) * np.pi / (2 * nodes))      # Chebyshev nodes of [0, 1]
    f = target(x)
    V = np.vander(x, degree + 1)                                    # highest power first
    w = np.ones(nodes)
    for _ in range(iters):
        sw = np.sqrt(w) / f                                         # relative-error weighting
        c, *_ = np.linalg.lstsq(V * sw[:, None], f * sw, rcond=None)
        err = np.abs(V @ c - f) / f
        w = w * err
        w /= w.sum()
    return c.astype(np.float32)


def horner_f32(c: np.ndarray, e: np.ndarray) -> np.ndarray:
    """e * q(e) evaluated as the kernel does: float32 Horner steps (fma
    rounding emulated by float64 products rounded to float32)."""
    e32 = np.asarray(e, np.float32)
    q = np.full_like(e32, c[0])
    for ci in c[1:]:
        q = (q.astype(np.float64) * e32.astype(np.float64) + np.float64(ci)).astype(np.float32)
    return (e32.astype(np.float64) * q.astype(np.float64)).astype(np.float32)


def max_rel_error(c: np.ndarray, n: int = 200001) -> float:
    """Largest relative error of e * q(e) against log1p(e) over (0, 1]."""
    e = np.linspace(1e-7, 1.0, n).astype(np.float32)
    ref = np.log1p(e.astype(np.float64))
    return float(np.max(np.abs(horner_f32(c, e) - ref) / ref))


if __name__ == "__main__":
    c = fit()
    print("coefficients, highest degree first:")
    for v in c:
        print(f"  {v!r}")
    print(f"max relative error of e*q(e) in float32: {max_rel_error(c):.3e}")

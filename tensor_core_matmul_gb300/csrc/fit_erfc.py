"""Fits the polynomial of the kernel's complementary error function.

The GPU's GELU needs erfc(z) for z >= 0 with a small relative error, in a
form without branches so that the 32 values a thread holds can be evaluated
side by side.  It uses the form of Press, Teukolsky, Vetterling and Flannery,
"Numerical Recipes" (2nd ed., section 6.2, the Chebyshev-fitted erfc):

    erfc(z) = t * exp(-z^2 + P(t)),   t = 1 / (1 + z/2),

where P is a polynomial; as z runs over [0, inf), t runs over (0, 1] and
P(t) = log(erfcx(z) / t) (erfcx(z) = exp(z^2) erfc(z)) is smooth on [0, 1].
This script computes P's coefficients itself: a least-squares fit in the
Chebyshev basis at Chebyshev nodes on [0, 1], converted to powers of t.  It
prints them as the C initialiser that gemm_kernel.cuh holds, and the largest
relative error of erfc over z in [0, 30] in double precision.

Run:  python tensor_core_matmul_gb300/csrc/fit_erfc.py
"""
from __future__ import annotations

import numpy as np

DEGREE = 9
NODES = 4000


def target(t: np.ndarray) -> np.ndarray:
    from scipy.special import erfcx
    z = 2.0 * (1.0 - t) / t
    return np.log(erfcx(z) / t)


def fit(degree: int = DEGREE) -> np.ndarray:
    """Coefficients c[0..degree] of P(t) = sum c[k] t^k."""
    n = NODES
    t = 0.5 * (1.0 - np.cos(np.pi * (np.arange(n) + 0.5) / n))  # Chebyshev nodes on [0, 1]
    t = np.clip(t, 1e-9, 1.0)
    cheb = np.polynomial.chebyshev.chebfit(2.0 * t - 1.0, target(t), degree)
    in_u = np.polynomial.Polynomial(np.polynomial.chebyshev.cheb2poly(cheb))  # powers of u = 2t - 1
    return in_u(np.polynomial.Polynomial([-1.0, 2.0])).coef


def max_rel_error(coef: np.ndarray) -> float:
    from scipy.special import erfc
    z = np.linspace(0.0, 30.0, 300001)
    t = 1.0 / (1.0 + 0.5 * z)
    approx = t * np.exp(-z * z + np.polynomial.polynomial.polyval(t, coef))
    exact = erfc(z)
    m = exact > 1e-300
    return float(np.max(np.abs(approx[m] - exact[m]) / exact[m]))


def c_initialiser(coef: np.ndarray) -> str:
    return "{" + ", ".join(f"{np.float32(c)!r}f".replace("np.float32(", "").replace(")", "") for c in coef) + "}"


if __name__ == "__main__":
    c = fit()
    print(c_initialiser(c))
    print(f"max relative error of erfc on [0, 30]: {max_rel_error(c):.3e}")

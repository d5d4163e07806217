"""Coefficients of the polynomial P(t) ~ log(1 + t) / t on [0, 1] used by the d = 128
kernels' front-end (``log1p_01`` in tc_util.cuh): a degree-7 least-squares fit on
Chebyshev nodes of [0, 1], in float64, printed highest power first as float32 literals.
Run ``python fit_log1p.py`` to regenerate; it also prints the fit's worst relative error
over a dense grid of [0, 1] (about 2e-7)."""

import numpy as np

DEGREE = 7
NODES = 4000


def fit():
    x = 0.5 * (1.0 - np.cos(np.pi * (np.arange(NODES) + 0.5) / NODES))
    return np.polyfit(x, np.log1p(x) / x, DEGREE)


def worst_relative_error(c):
    t = np.linspace(1e-9, 1.0, 400001)
    p = np.polyval(np.asarray(c, dtype=np.float64), t)
    return float(np.max(np.abs(t * p - np.log1p(t)) / np.log1p(t)))


if __name__ == "__main__":
    c = fit()
    c32 = c.astype(np.float32)
    print(", ".join(f"{v:.9e}f" for v in c32))
    print("worst relative error (float32 coefficients):", worst_relative_error(c32))

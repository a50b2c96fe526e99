"""Coefficients of the cubic that approximates 2^f on [-1/2, 1/2] in the dense prefix kernel.

The softmax of the dense kernel computes a quarter of its exponentials on the FMA pipe:
2^x = 2^j * 2^f with j = rint(x) and f = x - j in [-1/2, 1/2], and 2^f ~ c0 + c1 f + c2 f^2 +
c3 f^3.  The coefficients minimise the largest relative error max |p(f) / 2^f - 1| over a
dense grid of f (a Chebyshev / minimax fit), posed as a linear program:
    minimise t  subject to  -t <= (p(f_i) - 2^f_i) / 2^f_i <= t  for every grid point f_i.

  python -m shared_prefix_kv_decode_gb300.exp2_poly_fit [--degree 3]
"""

from __future__ import annotations

import argparse

import numpy as np


def fit(degree: int = 3, n: int = 4097):
    """Minimax coefficients (c0 .. c_degree, float64) and the fit's max relative error."""
    from scipy.optimize import linprog

    f = np.linspace(-0.5, 0.5, n)
    y = np.exp2(f)
    a = np.vstack([f ** k for k in range(degree + 1)]).T / y[:, None]
    nc = degree + 1
    cost = np.zeros(nc + 1)
    cost[-1] = 1.0
    a_ub = np.block([[a, -np.ones((n, 1))], [-a, -np.ones((n, 1))]])
    b_ub = np.concatenate([np.ones(n), -np.ones(n)])
    res = linprog(cost, A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * nc + [(0, None)], method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    return res.x[:nc], float(res.x[-1])


def eval_f32(coef, x):
    """The kernel's evaluation of 2^x in float32 arithmetic: clamp, round-to-nearest by adding
    1.5 * 2^23, Horner on f, exponent-field insertion."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0))
    rnd = np.float32(12582912.0)
    t = (x + rnd).astype(np.float32)
    f = (x - (t - rnd).astype(np.float32)).astype(np.float32)
    c = [np.float32(v) for v in coef]
    q = np.full_like(f, c[-1])
    for k in range(len(c) - 2, -1, -1):
        q = (q * f + c[k]).astype(np.float32)
    bits = q.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--degree", type=int, default=3)
    a = ap.parse_args(argv)
    coef, err = fit(a.degree)
    print("coefficients c0..c%d (float32):" % a.degree, [float(np.float32(c)) for c in coef])
    print("max relative error of the fit: %.3e" % err)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())

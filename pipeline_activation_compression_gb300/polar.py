"""PolarExpress polynomial coefficients for the SPEL step.

MAPL (§3.3, eqs. (6)-(7); App. E.4; Table 8) runs PolarExpress twice per
projector update -- 5 iterations for the spectral-norm LMO direction and 5 or 7
for the retraction onto St(d, r) -- but prints no coefficients.  This module
derives them with the method of Amsel, Persson, Musco and Gower, *The Polar
Express: Optimal Matrix Sign Methods and Their Application to the Muon
Algorithm* (ICLR 2026): iteration t uses the odd quintic p_t(x) = a x + b x^3 +
c x^5 that minimises max |1 - p(x)| over the interval [l_t, u_t] known to hold
the singular values; the next interval is the image [min p_t, max p_t] =
[1 - E_t, 1 + E_t], where E_t is the minimax error.  The minimax problem is
solved here with a Remez exchange on the 4-point alternation set {l, x1, x2, u}
(x1, x2 the interior critical points of p).

The table is a hyperparameter *input*: the CUDA library and the fp64 oracle
both receive the same (a, b, c) list.  Each iteration applies
Y <- Y (a I + b S + c S^2) with S = Y^T Y.
"""
from __future__ import annotations

import numpy as np

__all__ = ["minimax_odd_quintic", "polar_express_schedule", "default_coeffs",
           "NEWTON_SCHULZ_QUINTIC"]

#: limit of the schedule as the interval shrinks to {1}: p(1)=1, p'(1)=p''(1)=0
NEWTON_SCHULZ_QUINTIC = (15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0)


def _solve(xs):
    # a x + b x^3 + c x^5 + s_i E = 1 at the four alternation points
    s = np.array([1.0, -1.0, 1.0, -1.0])
    M = np.stack([xs, xs ** 3, xs ** 5, s], axis=1)
    a, b, c, E = np.linalg.solve(M, np.ones(4))
    return a, b, c, E


def _critical(a, b, c, lo, hi):
    # p'(x) = a + 3b x^2 + 5c x^4 = 0, a quadratic in y = x^2
    ys = np.roots([5.0 * c, 3.0 * b, a]) if c != 0 else np.roots([3.0 * b, a])
    xs = sorted(float(np.sqrt(y.real)) for y in ys
                if abs(y.imag) < 1e-12 and y.real > 0 and lo < np.sqrt(y.real) < hi)
    return xs


def minimax_odd_quintic(lo: float, hi: float, iters: int = 100, tol: float = 1e-15):
    """(a, b, c, E): the odd quintic closest to 1 in max norm on [lo, hi],
    0 < lo < hi, and its error E = max |1 - p(x)| on that interval."""
    if not (0.0 < lo < hi):
        raise ValueError("need 0 < lo < hi")
    # Chebyshev-like initial alternation set
    t = np.cos(np.pi * np.arange(3, -1, -1) / 3.0)
    xs = lo + (hi - lo) * (t + 1.0) / 2.0
    a = b = c = E = 0.0
    for _ in range(iters):
        a, b, c, E = _solve(xs)
        crit = _critical(a, b, c, lo, hi)
        if len(crit) != 2:
            break
        new = np.array([lo, crit[0], crit[1], hi])
        if np.max(np.abs(new - xs)) < tol * hi:
            xs = new
            break
        xs = new
    a, b, c, E = _solve(xs)
    grid = np.concatenate([np.linspace(lo, hi, 20001), xs])
    err = np.max(np.abs(1.0 - (a * grid + b * grid ** 3 + c * grid ** 5)))
    return float(a), float(b), float(c), float(err)


def polar_express_schedule(n: int, lo: float, hi: float = 1.0):
    """n per-iteration (a, b, c) coefficient triples starting from the
    singular-value interval [lo, hi]."""
    out = []
    for _ in range(n):
        if hi - lo < 1e-7:
            out.append(NEWTON_SCHULZ_QUINTIC)
            continue
        a, b, c, E = minimax_odd_quintic(lo, hi)
        out.append((a, b, c))
        lo, hi = max(1.0 - E, 1e-12), 1.0 + E
    return out


def default_coeffs(n_lmo: int = 5, n_retr: int = 5, lmo_lo: float = 1e-3,
                   retr_halfwidth: float = 0.1) -> np.ndarray:
    """(n_lmo + n_retr) x 3 float32 table: LMO rows first, then retraction.

    LMO: input scaled by its Frobenius norm, so singular values lie in (0, 1];
    those below ``lmo_lo`` are only partly mapped to 1.  Retraction: input
    A - alpha d has singular values close to 1; the schedule starts from
    [1 - retr_halfwidth, 1 + retr_halfwidth].
    """
    lmo = polar_express_schedule(n_lmo, lmo_lo, 1.0)
    retr = polar_express_schedule(n_retr, 1.0 - retr_halfwidth, 1.0 + retr_halfwidth)
    return np.asarray(lmo + retr, dtype=np.float32).reshape(n_lmo + n_retr, 3)

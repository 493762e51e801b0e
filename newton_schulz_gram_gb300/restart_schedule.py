"""Choosing when to restart Gram Newton-Schulz (Dion3 App. B.2.1).

Half-precision rounding leaves the Gram matrix R with small spurious negative
eigenvalues, which the polynomial iteration amplifies in Q_t. Restarting
(X <- Q X, R <- X X^T, Q <- I) removes them, at the cost of two rectangular
products. For a given coefficient schedule and number of restarts, the
appendix simulates the iteration on the eigenvalues of R (Theorem 2: each
eigenvalue follows its own scalar recurrence), subtracts a corruption of
4e-4 from R at every restart, and picks the schedule that minimizes the
largest condition number of Q_t over the steps.

This module restates that search. Its result feeds
`gns_orthogonalize_batched_schedule` (bit t of the mask: restart after
step t).
"""
from __future__ import annotations

import itertools

import numpy as np

QUINTIC = (3.4445, -4.7750, 2.0315)


def _schedule(coeffs, steps):
    if coeffs is None:
        return [QUINTIC] * steps
    coeffs = [tuple(map(float, c)) for c in coeffs]
    if len(coeffs) != steps:
        raise ValueError("one (a, b, c) per step")
    return coeffs


def simulate(coeffs=None, steps=5, restarts=(), lo=-4e-4, hi=1.0, points=4001, corruption=4e-4):
    """Scalar Gram NS over the eigenvalues of R_0 in [lo, hi] (Theorem 2):
    z_t = a_t + b_t r + c_t r^2, q_t = q_{t-1} z_t, r_t = r_{t-1} z_t^2.

    Each eigen-direction carries a true value (a squared singular value of
    the current X, never negative); the computed R is the true value minus
    `corruption`, as for R_0 (true value r_0 + corruption). A restart after
    step s multiplies the true value by q_s^2 (X <- Q X), recomputes
    r = true - corruption and resets q to 1.

    Returns the largest condition number of Q_t over all steps (max |q| / min
    |q| over the eigenvalues), the largest |q_t|, the smallest r_t, and the
    overall gain x_T / x_0 per eigenvalue."""
    sched = _schedule(coeffs, steps)
    r0 = np.linspace(lo, hi, points)
    true = r0 + corruption  # true value at the last (re)start
    r = r0.copy()
    q = np.ones_like(r0)
    gain = np.ones_like(r0)
    rs = set(int(t) for t in restarts)
    worst_cond, worst_q, min_r = 1.0, 1.0, float(r.min())
    with np.errstate(over="ignore", invalid="ignore"):
        for t, (a, b, c) in enumerate(sched, start=1):
            if (t - 1) in rs and t > 1:
                gain = gain * q
                true = q * q * true
                r = true - corruption
                q = np.ones_like(r0)
            z = a + b * r + c * r * r
            q = q * z
            r = r * z * z
            aq = np.abs(q)
            worst_cond = max(worst_cond, float(aq.max() / max(aq.min(), 1e-300)))
            worst_q = max(worst_q, float(aq.max()))
            min_r = min(min_r, float(r.min()))
    return {"max_cond_q": worst_cond, "max_q": worst_q, "min_r": min_r, "gain": gain * q, "r0": r0}


def best_schedule(coeffs=None, steps=5, n_restarts=1, **kw):
    """The restart steps (a tuple) among all choices of n_restarts steps in
    1 .. steps - 1 with the smallest largest condition number of Q_t, and that
    number."""
    best = None
    for cand in itertools.combinations(range(1, steps), n_restarts):
        v = simulate(coeffs, steps, cand, **kw)["max_cond_q"]
        if best is None or v < best[1]:
            best = (cand, v)
    return best


def restart_mask(restarts):
    """Bit t set: restart after step t."""
    m = 0
    for t in restarts:
        m |= 1 << int(t)
    return m

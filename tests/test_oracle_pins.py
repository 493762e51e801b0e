"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each expected value comes from
an independent route (a closed form via a library SVD, Theorem 2's scalar
composition, FLOP formulas printed on the pages, invariances).
"""
import os

import numpy as np
import pytest

from inputs import generators as gen
from oracle import gram_ns as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PAGES_TEST_COEFFS = (15 / 8, -10 / 8, 3 / 8)  # Dion3 App. B.1.1


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def svd_closed_form(X, steps, coeffs):
    """Closed form of any NS variant in exact arithmetic (Dion3 §2.2 and
    Theorem 2): X = U S V^T  ->  U p(S_hat) V^T with S_hat = S / (1.05 (||X||_F + eps))
    and p the composed odd polynomial. Uses numpy's SVD, not the oracle."""
    U, S, Vt = np.linalg.svd(np.asarray(X, np.float64), full_matrices=False)
    s_hat = S / (1.05 * (np.linalg.norm(X) + 1e-7))
    ps = s_hat.copy()
    for a, b, c in O.coeff_schedule(steps, coeffs):
        ps = a * ps + b * ps ** 3 + c * ps ** 5
    return (U * ps) @ Vt


# ---------------------------------------------------------------- constants

def test_quintic_matches_page():
    vals = [l for l in open(os.path.join(GOLDEN, "quintic.txt")) if not l.startswith("#")]
    a, b, c = (float(v) for v in vals[0].split())
    assert O.QUINTIC == (a, b, c)
    assert O.SAFETY == 1.05 and O.EPS == 1e-7


# ------------------------------------------------------------------ Theorem 2

@pytest.mark.parametrize("coeffs", [None, PAGES_TEST_COEFFS, "random"])
@pytest.mark.parametrize("steps", [1, 3, 5, 8])
def test_theorem2_scalar_recurrence_equals_composition(coeffs, steps):
    if coeffs == "random":
        # Arbitrary per-step coefficients, kept small enough that nothing overflows.
        coeffs = np.random.default_rng(steps).uniform(-0.6, 0.9, size=3 * steps)
    x = np.linspace(0.0, 1.0, 257)
    direct = O.compose_odd_polys(x, steps, coeffs)
    via_q = O.scalar_gram_recurrence(x, steps, coeffs) * x
    assert np.all(np.isfinite(direct))
    np.testing.assert_allclose(via_q, direct, rtol=1e-12, atol=1e-13)


def test_scalar_recurrence_known_value():
    # One step of the quintic at x = 0.5: q_1 = a + b/4 + c/16.
    a, b, c = O.QUINTIC
    assert O.scalar_gram_recurrence(np.array([0.5]), 1)[0] == pytest.approx(a + b / 4 + c / 16, rel=1e-15)


# ------------------------------------------------------ spectral action (SVD)

SHAPES = [(8, 32), (16, 48), (40, 12), (5, 5), (3, 64)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("variant", ["standard", "naive", "restart2", "restart1", "norestart"])
def test_spectral_action_matches_svd_closed_form(shape, variant):
    X = gen.gaussian(*shape, seed=11, index=hash(shape) % 1000).astype(np.float64)
    if variant == "standard":
        out = O.standard_ns(X)
    elif variant == "naive":
        out = O.gram_ns_naive(X)
    else:
        ra = {"restart2": 2, "restart1": 1, "norestart": 0}[variant]
        out = O.gram_ns(X, restart_at=ra)
    expect = svd_closed_form(X, 5, None)
    assert rel(out, expect) < 1e-11


@pytest.mark.parametrize("shape", [(8, 32), (24, 10)])
def test_singular_vectors_unchanged(shape):
    X = gen.gaussian(*shape, seed=12).astype(np.float64)
    out = O.gram_ns(X)
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    # U^T out V must be diagonal: the iteration acts on singular values only.
    D = U.T @ out @ Vt.T
    off = D - np.diag(np.diag(D))
    assert np.linalg.norm(off) < 1e-12 * np.linalg.norm(D)


# ------------------------------------------------- Gram NS == standard NS

def test_gram_equals_standard_on_128x512():
    X = gen.gaussian(128, 512, seed=1000, index=0).astype(np.float64)
    std = O.standard_ns(X)
    for out in (O.gram_ns(X), O.gram_ns_naive(X), O.gram_ns(X, restart_at=1)):
        assert rel(out, std) < 1e-12


def test_restart_every_step_is_standard_ns():
    X = gen.gaussian(48, 160, seed=3).astype(np.float64)
    assert rel(O.gram_ns(X, restart_at=1, steps=7), O.standard_ns(X, steps=7)) < 1e-13


def test_restart_schedule():
    assert O.restart_points(5, 2) == [2]
    assert O.restart_points(25, 5) == [5, 10, 15, 20]
    assert O.restart_points(5, 1) == [1, 2, 3, 4]
    assert O.restart_points(5, 0) == []
    assert O.restart_points(5, 5) == []
    assert O.restart_points(10, 3) == [3, 6]


# --------------------------------------------------- convergence to polar

def test_converges_to_polar_with_restarts():
    """With the textbook quintic (15/8, -10/8, 3/8) (Dion3 App. B.1) and
    restarts every 5 steps (App. B.2), a well-conditioned input converges to
    polar(X) = U V^T (Definition 1)."""
    r = np.random.default_rng(5)
    U = gen.orthonormal_rows(16, 16, r)
    V = gen.orthonormal_rows(16, 64, r)
    s = r.uniform(0.1, 1.0, size=16)
    X = (U * s) @ V
    out = O.gram_ns(X, steps=20, coeffs=PAGES_TEST_COEFFS, restart_at=5)
    assert rel(out, U @ V) < 1e-12
    out_std = O.standard_ns(X, steps=20, coeffs=PAGES_TEST_COEFFS)
    assert rel(out_std, U @ V) < 1e-12


def test_equal_singular_values_give_scaled_input():
    """Orthonormal rows: every normalized singular value is 1/(1.05 (sqrt(n)+eps)),
    so the output is exactly kappa * X with kappa = p(sigma_hat) (Theorem 2)."""
    X = gen.orthonormal_rows_matrix(32, 128, seed=9, dtype=np.float64)
    n = 32
    s_hat = 1.0 / (1.05 * (np.linalg.norm(X) + 1e-7))
    assert np.linalg.norm(X) == pytest.approx(np.sqrt(n), rel=1e-12)
    kappa = O.compose_odd_polys(np.array([s_hat]))[0]
    for out in (O.gram_ns(X), O.standard_ns(X), O.gram_ns_naive(X)):
        assert rel(out, kappa * X) < 1e-12


# -------------------------------------------------------------- symmetry

def test_gram_state_is_symmetric():
    X = gen.gaussian(64, 256, seed=21).astype(np.float64)
    trace = []
    O.gram_ns(X, trace=trace)
    names = {name for _, name, _ in trace}
    assert {"R", "Z", "Q", "RZ"} <= names
    for t, name, M in trace:
        if name == "X":
            continue
        assert np.linalg.norm(M - M.T) <= 1e-13 * np.linalg.norm(M), (t, name)


def test_trace_follows_algorithm3_order():
    """Algorithm 3 at T = 5 with a restart after step 2 computes, in order:
    R0; t1 Z,Q,RZ,R; t2 Z,Q; restart X,R; t3 Z,Q,RZ,R; t4 Z,Q,RZ,R; t5 Z,Q."""
    trace = []
    O.gram_ns(gen.gaussian(8, 24, seed=1).astype(np.float64), trace=trace)
    seq = [(t, n) for t, n, _ in trace]
    assert seq == [(0, "R"), (1, "Z"), (1, "Q"), (1, "RZ"), (1, "R"), (2, "Z"), (2, "Q"),
                   (3, "X"), (3, "R"), (3, "Z"), (3, "Q"), (3, "RZ"), (3, "R"),
                   (4, "Z"), (4, "Q"), (4, "RZ"), (4, "R"), (5, "Z"), (5, "Q")]


# ------------------------------------------------------------- FLOP counts

@pytest.mark.parametrize("n,alpha", [(16, 1), (16, 4), (8, 3), (32, 2)])
@pytest.mark.parametrize("T", [3, 5])
def test_flop_counts_match_page_formulas(n, alpha, T):
    m = alpha * n
    X = gen.gaussian(n, m, seed=2).astype(np.float64)

    c = O.FlopCounter(symmetric_products=False)
    O.standard_ns(X, steps=T, counter=c)
    assert c.flops == 2 * T * (2 * alpha + 1) * n ** 3  # Dion3 §2.2
    assert c.products == 3 * T

    c = O.FlopCounter()
    O.standard_ns(X, steps=T, counter=c)
    assert c.flops == T * (3 * alpha + 1) * n ** 3  # Dion3 §2.3

    c = O.FlopCounter()
    O.gram_ns_naive(X, steps=T, counter=c)
    assert c.flops == (4 * T + 3 * alpha - 3) * n ** 3  # Dion3 §4.1

    c = O.FlopCounter()
    O.gram_ns(X, steps=T, restart_at=2, counter=c)
    restarts = len(O.restart_points(T, 2))
    assert c.flops == O.flops_gram_restarted(n, m, T, restarts)
    if T == 5:
        assert c.flops == (4 * T + 6 * alpha - 6) * n ** 3  # blog post, FLOP section


def test_flop_ratios_printed_on_pages():
    n, alpha, T = 64, 4, 5
    m = alpha * n
    plain = O.flops_standard_plain(n, m, T)
    sym = O.flops_standard_symmetric(n, m, T)
    naive = O.flops_gram_naive(n, m, T)
    restarted = O.flops_gram_restarted(n, m, T)
    got = {("naive_gram", "standard_symmetric"): 1 - naive / sym,
           ("naive_gram", "standard_plain"): 1 - naive / plain,
           ("restarted_gram", "standard_symmetric"): 1 - restarted / sym}
    rows = [l.split() for l in open(os.path.join(GOLDEN, "flop_ratios.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for variant, base, pct, *_ in rows:
        assert round(100 * got[(variant, base)]) == int(pct)


# ------------------------------------------------------------- invariances

def test_scale_invariance():
    X = gen.gaussian(24, 80, seed=4).astype(np.float64)
    base = O.gram_ns(X)
    for s in (1e-3, 1e3):
        # eps = 1e-7 against ||sX||_F ~ s*44 moves the result by < 1e-5 relative.
        assert rel(O.gram_ns(s * X), base) < 1e-5


def test_transpose_equivariance():
    X = gen.gaussian(20, 70, seed=5).astype(np.float64)
    assert np.array_equal(O.orthogonalize(X.T), O.orthogonalize(X).T)


def test_zero_maps_to_zero():
    for shape in ((8, 32), (16, 16)):
        out = O.orthogonalize(np.zeros(shape))
        assert np.all(out == 0) and np.all(np.isfinite(out))


# --------------------------------------- finite-precision diagnostic (App. B)

def _lowp(x, dtype):
    return np.asarray(x, dtype=np.float32).astype(dtype).astype(np.float64)


def _naive_lowp(X, steps, coeffs, dtype):
    """Algorithm 2 with every stored matrix rounded to ``dtype`` (products
    accumulate in fp64 here; the rounding of stored values is what matters)."""
    X = _lowp(O.normalize(X), dtype)
    n = X.shape[0]
    R = _lowp(X @ X.T, dtype)
    Q = np.eye(n)
    hist = []
    for a, b, c in O.coeff_schedule(steps, coeffs):
        Z = _lowp(a * np.eye(n) + b * R + c * (R @ R), dtype)
        Q = _lowp(Q @ Z, dtype)
        R = _lowp(Z @ _lowp(R @ Z, dtype), dtype)
        hist.append(np.linalg.eigvalsh(R).min())
    return Q @ X, hist


def test_naive_gram_develops_negative_eigenvalues_in_half_precision():
    """Dion3 App. B.1: in half precision, R_t of naive Gram NS develops
    negative eigenvalues that grow (r_t < 0 diverges, Fig. 13), while the
    fp64 iteration keeps R_t positive semidefinite."""
    X = gen.exp_decay_spectrum(128, 512, seed=6, decay=0.1)
    _, hist16 = _naive_lowp(X, 10, PAGES_TEST_COEFFS, np.float16)
    trace = []
    O.gram_ns(X, steps=10, coeffs=PAGES_TEST_COEFFS, restart_at=0, trace=trace)
    min64 = min(np.linalg.eigvalsh(M).min() for t, n, M in trace if n == "R")
    assert min64 > -1e-12
    assert hist16[-1] < -1e-3 and hist16[-1] < 10 * min(hist16[:3])

"""fp64 CPU oracle for (Gram) Newton-Schulz orthogonalization.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may import
this module. The library under ``newton_schulz_gram_gb300/`` never does, and
shares no code with it.

What it computes, and where each step comes from. All citations are to
"Dion3: Full-stack orthogonal updates" (arXiv 2608.11612) unless noted.

* ``standard_ns``: the quintic Newton-Schulz iteration of §2.2, Algorithm 1:
  A = X X^T, B = b A + c A^2, X <- a X + B X, repeated T times.
* ``gram_ns_naive``: Algorithm 2 of §4. Iterates on the n x n Gram matrix
  R = X X^T with Z = a I + b R + c R^2, Q <- Q Z, R <- Z R Z, returns Q X.
* ``gram_ns``: the stabilized form of §4.2, Algorithm 3. The a-term is
  distributed over the later products as App. B.2.3 describes
  (Z = b R + c R^2, Q <- Q Z + a Q, RZ <- R Z + a R, R <- Z RZ + a RZ), and the
  iteration restarts (X <- Q X, R <- X X^T, Q <- I).
* Safety factor: the input is scaled once to Frobenius norm 1/1.05
  (App. B.2.2 recommends 1.05 over 1.02).
* ``scalar_gram_recurrence``: Theorem 2, the scalar iteration
  r_0 = x^2, q_0 = 1, z = h(r), r <- r z^2, q <- q z.
* FLOP accounting (``FlopCounter``): §2.2 and §2.3 (standard NS with and
  without symmetric products), §4.1 (naive Gram NS). The restarted total
  (4T + 6 alpha - 6) n^3 is stated on the third page (Gram Newton-Schulz
  blog post, section "FLOP" comparison).

Readings where the pages leave a step open:

* Transposition: a matrix with more rows than columns is transposed first, so
  X is n x m with n <= m, and transposed back at the end (§2.2 assumes n <= m;
  the grouped Muon kernel card, "How it works", transposes so the contracted
  dimension is the larger one).
* Normalization: X / (1.05 * (||X||_F + 1e-7)). An all-zero input gives an
  all-zero output.
* Restart schedule: ``restart_at = p`` restarts after every step t with
  t % p == 0 and at least p steps left (T - t >= p). For T = 5, p = 2 this is
  the single restart after step 2 of Algorithm 3; for p = 1 it restarts after
  every step, which is standard NS; p <= 0 never restarts.
* Square matrices: the pages fall back to standard NS (§4.1, last
  paragraph); all variants agree in exact arithmetic.
"""
from __future__ import annotations

import numpy as np

# Constant quintic of the grouped Muon kernel card ("How it works").
QUINTIC = (3.4445, -4.7750, 2.0315)
# Safety factor recommended in App. B.2.2.
SAFETY = 1.05
# Normalization epsilon of Algorithms 1-3, line 2.
EPS = 1e-7


def coeff_schedule(steps, coeffs=None):
    """Per-step (a_t, b_t, c_t) list. ``coeffs`` is None (constant quintic),
    one triple (used at every step), or a flat/nested sequence of 3*steps."""
    if steps < 1:
        raise ValueError("steps must be >= 1")
    if coeffs is None:
        return [tuple(float(v) for v in QUINTIC)] * steps
    arr = np.asarray(coeffs, dtype=np.float64).reshape(-1)
    if arr.size == 3:
        return [tuple(arr.tolist())] * steps
    if arr.size != 3 * steps:
        raise ValueError("coeffs must hold 3 or 3*steps values")
    return [tuple(arr[3 * t:3 * t + 3].tolist()) for t in range(steps)]


def restart_points(steps, restart_at):
    """Steps t (1-based) after which the Gram iteration restarts: every
    multiple of the period restart_at with at least one period left, or an
    explicit list of steps (any schedule, Dion3 App. B.2.1 sweeps them)."""
    if isinstance(restart_at, (list, tuple, set, frozenset)):
        return sorted(t for t in set(restart_at) if 1 <= t < steps)
    if restart_at is None or restart_at <= 0:
        return []
    return [t for t in range(1, steps) if t % restart_at == 0 and steps - t >= restart_at]


class FlopCounter:
    """Counts the FLOPs of the cubic-time products only (§2.2 counts only
    matrix multiplications). A general product of (M x K)(K x N) costs
    2 M N K. A product whose result is symmetric costs half of that when the
    caller asks for the symmetric count (§2.3: computing only the lower
    triangle halves the cost)."""

    def __init__(self, symmetric_products=True):
        self.symmetric_products = symmetric_products
        self.flops = 0
        self.products = 0

    def mm(self, A, B, symmetric=False):
        m, k = A.shape
        k2, n = B.shape
        assert k == k2
        cost = 2 * m * n * k
        if symmetric and self.symmetric_products:
            cost //= 2
        self.flops += cost
        self.products += 1
        return A @ B


def _mm(counter, A, B, symmetric=False):
    if counter is None:
        return A @ B
    return counter.mm(A, B, symmetric)


def orient(X):
    """Return (X', transposed) with X' having no more rows than columns."""
    X = np.asarray(X, dtype=np.float64)
    if X.ndim != 2:
        raise ValueError("expected a 2D matrix")
    if X.shape[0] > X.shape[1]:
        return X.T.copy(), True
    return X.copy(), False


def normalize(X):
    """Line 2 of Algorithms 1-3 plus the 1.05 safety factor (App. B.2.2)."""
    return X / (SAFETY * (np.linalg.norm(X, "fro") + EPS))


def standard_ns(X, steps=5, coeffs=None, counter=None):
    """Algorithm 1 (§2.2): standard quintic Newton-Schulz in fp64."""
    X, transposed = orient(X)
    X = normalize(X)
    for a, b, c in coeff_schedule(steps, coeffs):
        A = _mm(counter, X, X.T, symmetric=True)
        B = b * A + c * _mm(counter, A, A, symmetric=True)
        X = a * X + _mm(counter, B, X)
    return X.T if transposed else X


def gram_ns_naive(X, steps=5, coeffs=None, counter=None):
    """Algorithm 2 (§4): naive Gram Newton-Schulz in fp64.

    Q_1 = Q_0 Z_1 = Z_1 costs nothing since Q_0 = I, and R_T is never used,
    so neither is computed (§4.1)."""
    X, transposed = orient(X)
    X = normalize(X)
    n = X.shape[0]
    I = np.eye(n)
    R = _mm(counter, X, X.T, symmetric=True)
    Q = None  # identity
    sched = coeff_schedule(steps, coeffs)
    for t, (a, b, c) in enumerate(sched, start=1):
        Z = a * I + b * R + c * _mm(counter, R, R, symmetric=True)
        Q = Z if Q is None else _mm(counter, Q, Z, symmetric=True)
        if t < steps:
            ZR = _mm(counter, Z, R, symmetric=True)
            R = _mm(counter, ZR, Z, symmetric=True)
    out = _mm(counter, Q, X)
    return out.T if transposed else out


def gram_ns(X, steps=5, coeffs=None, restart_at=2, counter=None, trace=None):
    """Algorithm 3 (§4.2) with the a-term distribution of App. B.2.3.

    ``trace``, when a list, receives (t, name, matrix) for every Gram-state
    matrix computed, so tests can inspect R, Q, Z and RZ."""
    X, transposed = orient(X)
    X = normalize(X)
    n = X.shape[0]
    I = np.eye(n)
    sched = coeff_schedule(steps, coeffs)
    restarts = set(restart_points(steps, restart_at))

    R = _mm(counter, X, X.T, symmetric=True)
    Q = None  # identity; the first Q after a (re)start is Z + a I
    if trace is not None:
        trace.append((0, "R", R))
    for t, (a, b, c) in enumerate(sched, start=1):
        if (t - 1) in restarts:
            X = _mm(counter, Q, X)
            R = _mm(counter, X, X.T, symmetric=True)
            Q = None
            if trace is not None:
                trace.append((t, "X", X))
                trace.append((t, "R", R))
        Z = b * R + c * _mm(counter, R, R, symmetric=True)
        if Q is None:
            Q = Z + a * I
        else:
            Q = _mm(counter, Q, Z, symmetric=True) + a * Q
        if trace is not None:
            trace.append((t, "Z", Z))
            trace.append((t, "Q", Q))
        # R_t is needed only if another step follows without a restart.
        if t < steps and t not in restarts:
            RZ = _mm(counter, R, Z, symmetric=True) + a * R
            R = _mm(counter, Z, RZ, symmetric=True) + a * RZ
            if trace is not None:
                trace.append((t, "RZ", RZ))
                trace.append((t, "R", R))
    out = _mm(counter, Q, X)
    return out.T if transposed else out


def orthogonalize(X, steps=5, coeffs=None, restart_at=2):
    """What the library computes for one matrix: restarted Gram NS for a
    rectangular matrix, standard NS for a square one (§4.1, last paragraph)."""
    X = np.asarray(X, dtype=np.float64)
    if X.shape[0] == X.shape[1]:
        return standard_ns(X, steps, coeffs)
    return gram_ns(X, steps, coeffs, restart_at)


def orthogonalize_batched(Xs, steps=5, coeffs=None, restart_at=2):
    """Each matrix of a [G, R, C] stack on its own (the bucket is not an
    approximation: the grouped Muon kernel card, "Correctness")."""
    Xs = np.asarray(Xs, dtype=np.float64)
    return np.stack([orthogonalize(x, steps, coeffs, restart_at) for x in Xs])


# ----------------------------------------------------------------------------
# Scalar forms (Theorem 2) used to pin the matrix iterations.
# ----------------------------------------------------------------------------

def compose_odd_polys(x, steps=5, coeffs=None):
    """(p_T o ... o p_1)(x) with p_t(x) = a x + b x^3 + c x^5 (§2.2)."""
    x = np.asarray(x, dtype=np.float64)
    for a, b, c in coeff_schedule(steps, coeffs):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def scalar_gram_recurrence(x, steps=5, coeffs=None):
    """Theorem 2: returns q_T with (p_T o ... o p_1)(x) = q_T x, from
    r_0 = x^2, q_0 = 1, z_t = h_t(r_{t-1}), r_t = r_{t-1} z_t^2, q_t = q_{t-1} z_t,
    where h_t(y) = a_t + b_t y + c_t y^2."""
    x = np.asarray(x, dtype=np.float64)
    r = x * x
    q = np.ones_like(x)
    for a, b, c in coeff_schedule(steps, coeffs):
        z = a + b * r + c * r * r
        r = r * z * z
        q = q * z
    return q


# ----------------------------------------------------------------------------
# FLOP formulas as the pages state them (used by the FLOP pins and the bench).
# ----------------------------------------------------------------------------

def flops_standard_plain(n, m, steps=5):
    """§2.2: T (4 m n^2 + 2 n^3) = 2 T (2 alpha + 1) n^3."""
    return steps * (4 * m * n * n + 2 * n ** 3)


def flops_standard_symmetric(n, m, steps=5):
    """§2.3: T (3 alpha + 1) n^3 with symmetric products."""
    return steps * (3 * m * n * n + n ** 3)


def flops_gram_naive(n, m, steps=5):
    """§4.1: (4 T + 3 alpha - 3) n^3."""
    return 4 * steps * n ** 3 + 3 * m * n * n - 3 * n ** 3


def flops_gram_restarted(n, m, steps=5, restarts=1):
    """Each restart adds X <- Q X (2 alpha n^3) and R <- X X^T (alpha n^3) and
    removes the Q-product that Q = I makes free (n^3) and the R and RZ
    products of the step before it (2 n^3): 3 (alpha - 1) n^3 in all (§4.2).
    With one restart this is the (4 T + 6 alpha - 6) n^3 of the third page."""
    return flops_gram_naive(n, m, steps) + restarts * (3 * m * n * n - 3 * n ** 3)

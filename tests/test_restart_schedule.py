"""The restart-schedule search (Dion3 App. B.2.1) against the oracle's
scalar Gram recurrence (Theorem 2) and the appendix's qualitative findings."""
import numpy as np

from newton_schulz_gram_gb300 import restart_schedule as RS
from oracle import gram_ns as O


def test_restarts_change_nothing_in_exact_arithmetic():
    """With no corruption and no negative eigenvalues every schedule gives
    the same overall gain, and it is Theorem 2's q_T (the composed polynomial
    divided by x)."""
    x = np.sqrt(np.linspace(0.0, 1.0, 101))
    want = O.scalar_gram_recurrence(x, 5)
    for restarts in [(), (1,), (2,), (3,), (2, 3), (1, 2, 3, 4)]:
        d = RS.simulate(None, 5, restarts, lo=0.0, hi=1.0, points=101, corruption=0.0)
        assert np.allclose(d["gain"], want, rtol=1e-12), restarts
    coeffs = [(15 / 8, -10 / 8, 3 / 8)] * 10
    d = RS.simulate(coeffs, 10, (5,), lo=0.0, hi=1.0, points=101, corruption=0.0)
    assert np.allclose(d["gain"], O.scalar_gram_recurrence(x, 10, coeffs), rtol=1e-12)


def test_restarting_bounds_the_spurious_negative_eigenvalues():
    """Without a restart the eigenvalues of R_0 near -4e-4 make Q blow up;
    one restart keeps the largest |q| and cond(Q) bounded (App. B.2.1)."""
    none = RS.simulate(None, 5, ())
    after2 = RS.simulate(None, 5, (2,))
    assert none["max_q"] > 1e5 and none["min_r"] < -1e3
    assert after2["max_q"] < 1e2 and after2["min_r"] > -1.0
    long_none = RS.simulate([(15 / 8, -10 / 8, 3 / 8)] * 25, 25, ())
    long_every5 = RS.simulate([(15 / 8, -10 / 8, 3 / 8)] * 25, 25, (5, 10, 15, 20))
    assert not np.isfinite(long_none["max_q"]) or long_none["max_q"] > 1e10
    assert long_every5["max_q"] < 100


def test_best_schedule_is_the_minimum_over_all_candidates():
    best, val = RS.best_schedule(None, 5, 1)
    vals = {t: RS.simulate(None, 5, (t,))["max_cond_q"] for t in range(1, 5)}
    assert val == min(vals.values()) and vals[best[0]] == val
    best2, val2 = RS.best_schedule(None, 5, 2)
    assert len(best2) == 2 and val2 <= val * 1.0001  # a second restart never hurts here


def test_restart_mask():
    assert RS.restart_mask(()) == 0 and RS.restart_mask((2,)) == 4 and RS.restart_mask((1, 3)) == 10

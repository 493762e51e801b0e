"""The restarted iteration's own fp16 state on the GPU (Dion3 App. B.2.1,
Fig. 18): with a restart after step 2, the eigenvalues of R_t stay above
-0.4 and those of Q_t below about 100, for every step count. The state comes
from gns_gram_ns_state (the library's R and Q after the run, lower triangles,
R scaled by its power of two) and is also compared with the oracle's fp64
trace of the same schedule (Algorithm 3 with the App. B.2.3 a-terms).

The inputs include the cases the appendix worries about: a rank-32 matrix
(R_0 has hundreds of zero eigenvalues, which fp16 turns into spurious small
negative ones) and an exponentially decaying spectrum."""
import numpy as np
import pytest

from inputs import generators as gen
from oracle import gram_ns as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

R_MIN_BOUND = -0.4    # Fig. 18: eig(R_t) > -0.4 with a restart after step 2
Q_MAX_BOUND = 100.0   # Fig. 18: eig(Q_t) below about 100
STATE_TOL = 3e-2      # relative Frobenius error of the state against fp64


@pytest.fixture(scope="module")
def gns():
    import newton_schulz_gram_gb300 as m
    from newton_schulz_gram_gb300 import build
    build.build()
    m.load()
    return m


def bucket(rows, cols, seed):
    return np.stack([
        gen.gaussian(rows, cols, seed, 0),
        gen.low_rank(rows, cols, seed, 1, rank=32),
        gen.exp_decay_spectrum(rows, cols, seed, 2, decay=0.02).astype(np.float32),
        gen.student_t(rows, cols, seed, 3),
    ])


def sym_lower(a):
    a = np.asarray(a, dtype=np.float64)
    return np.tril(a) + np.tril(a, -1).T


def range_basis(x):
    """Orthonormal basis (n x k) of the range of the oriented, normalized X
    (the eigenvectors of the oracle's R_0 above 1e-10 of its largest
    eigenvalue): all of it for a full-rank input, 32 directions for a rank-32
    one. The Gram state is compared on this subspace; on the null space of
    an exactly rank-deficient X it holds only fp16 rounding noise amplified by
    the polynomial (the fp16 floor of low-rank inputs), which the eigenvalue
    bounds cover instead."""
    trace = []
    O.gram_ns(x.astype(np.float64), 1, None, [], trace=trace)
    w, v = np.linalg.eigh(trace[0][2])
    return v[:, w > 1e-10 * w.max()]


def rel_on(P, a, ref):
    return np.linalg.norm(P.T @ (a - ref) @ P) / np.linalg.norm(P.T @ ref @ P)


def oracle_state(x, steps, restarts):
    trace = []
    O.gram_ns(x.astype(np.float64), steps, None, list(restarts), trace=trace)
    r = [m for (_, name, m) in trace if name == "R"][-1]
    q = [m for (_, name, m) in trace if name == "Q"][-1]
    return r, q


@pytest.mark.parametrize("rows,cols", [(512, 2048), (2048, 512)], ids=["wide", "tall"])
def test_restarted_state_stays_bounded_and_matches_oracle(gns, rows, cols):
    X = bucket(rows, cols, seed=7300 + rows)
    bases = [range_basis(X[g]) for g in range(X.shape[0])]
    worst = {}
    for steps in range(1, 6):
        restarts = (2,) if steps >= 3 else ()
        t = torch.from_numpy(X.copy()).cuda()
        r_state, q_state, scale = gns.gns_gram_ns_state(t, steps, restarts)
        torch.cuda.synchronize()
        assert gns.gns_get_status() == 0
        assert scale > 0 and np.log2(scale) == int(np.log2(scale))
        r_all = r_state.float().cpu().numpy()
        q_all = q_state.float().cpu().numpy()
        for g in range(X.shape[0]):
            r = sym_lower(r_all[g]) / scale
            q = sym_lower(q_all[g])
            assert np.isfinite(r).all() and np.isfinite(q).all(), (steps, g)
            er, eq = np.linalg.eigvalsh(r), np.linalg.eigvalsh(q)
            assert er.min() > R_MIN_BOUND, (steps, g, er.min())
            assert eq.max() < Q_MAX_BOUND, (steps, g, eq.max())
            r_ref, q_ref = oracle_state(X[g], steps, restarts)
            rel_r, rel_q = rel_on(bases[g], r, r_ref), rel_on(bases[g], q, q_ref)
            full_r = np.linalg.norm(r - r_ref) / np.linalg.norm(r_ref)
            w = worst.setdefault(g, [0.0, 0.0, 0.0, np.inf, -np.inf])
            w[0], w[1], w[2] = max(w[0], rel_r), max(w[1], rel_q), max(w[2], full_r)
            w[3], w[4] = min(w[3], er.min()), max(w[4], eq.max())
            assert rel_r <= STATE_TOL and rel_q <= STATE_TOL, (steps, g, rel_r, rel_q)
    # Per matrix: worst R and Q error on the range, worst R error on the whole
    # space, lowest eigenvalue of R_t, highest of Q_t.
    print({g: [round(float(v), 5) for v in w] for g, w in worst.items()})


def test_state_entry_rejects_square_and_bad_masks(gns):
    x = torch.zeros(1, 64, 64, device="cuda")
    with pytest.raises(Exception):
        gns.gns_gram_ns_state(x, 5, (2,))
    x = torch.zeros(1, 64, 128, device="cuda")
    with pytest.raises(Exception):
        gns.gns_gram_ns_state(x, 5, (5,))

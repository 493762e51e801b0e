"""Pins of the Muon elementwise oracle: Philox known answers, the exactness
and unbiasedness of stochastic rounding, and closed forms of the momentum and
update arithmetic."""
import os

import numpy as np
import pytest

from inputs import generators as gen
from oracle import gram_ns as O_NS
from oracle import muon as MU

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answer_vectors():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for row in rows:
        v = [int(x, 16) for x in row]
        ctr, key, want = v[:4], v[4:6], v[6:]
        out = MU.philox4x32_10(*[np.array([c], np.uint32) for c in ctr], *key)
        assert [int(o[0]) for o in out] == want


def test_sr_keeps_representable_values():
    vals = np.array([0.0, -0.0, 1.0, -2.5, 3.140625, 2.0 ** -100, np.inf, -np.inf], np.float32)
    bits = vals.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0)
    out = MU.stochastic_round_bf16(vals, seed=1, step=2)
    assert np.array_equal(out.astype(np.uint32), bits >> 16)


def test_sr_nan_stays_nan():
    nan_low = np.array([0x7F800001], np.uint32).view(np.float32)  # payload only in low bits
    out = MU.stochastic_round_bf16(nan_low, 0, 0)
    assert np.isnan(MU.bf16_bits_to_f32(out))[0]


def test_sr_rounds_to_a_neighbour():
    rng = np.random.default_rng(0)
    w = (rng.standard_normal(50000) * 10 ** rng.uniform(-5, 5, 50000)).astype(np.float32)
    out = MU.stochastic_round_bf16(w, seed=7, step=3).astype(np.uint32)
    lo = w.view(np.uint32) >> 16
    assert np.all((out == lo) | (out == lo + 1))


def test_sr_reproducible_and_keyed():
    w = np.linspace(-3, 3, 4096, dtype=np.float32) + np.float32(1e-4)
    a = MU.stochastic_round_bf16(w, 5, 9)
    assert np.array_equal(a, MU.stochastic_round_bf16(w, 5, 9))
    assert not np.array_equal(a, MU.stochastic_round_bf16(w, 5, 10))
    assert not np.array_equal(a, MU.stochastic_round_bf16(w, 6, 9))


def test_sr_base_index_shards_round_identically():
    """The grouped Muon kernel card: base_index makes a matrix updated whole or
    in shards round identically."""
    w = np.random.default_rng(1).standard_normal(10007).astype(np.float32)
    whole = MU.stochastic_round_bf16(w, 3, 4, base_index=123)
    parts = np.concatenate([MU.stochastic_round_bf16(w[:4001], 3, 4, base_index=123),
                            MU.stochastic_round_bf16(w[4001:], 3, 4, base_index=123 + 4001)])
    assert np.array_equal(whole, parts)


@pytest.mark.parametrize("p", [0.1, 0.25, 0.5])
def test_sr_unbiased_subulp_update(p):
    """The grouped Muon kernel card: a sub-ULP update across 2e5 bf16 elements
    averages to the true value, where round-to-nearest leaves it unchanged.
    Mean over 16 (seed, step) draws of 2e5 elements: the sampling SD of the
    mean is sqrt(p(1-p)/3.2e6) <= 2.8e-4 ULP, so 1e-3 ULP is >= 3.5 SD."""
    n = 200_000
    ulp = np.float32(2.0 ** -7)  # bf16 ULP at 1.0
    w = np.full(n, np.float32(1.0) + np.float32(p) * ulp, np.float32)
    frac = (float(w[0]) - 1.0) / float(ulp)  # p as rounded into fp32
    errs = []
    for k in range(16):
        out = MU.bf16_bits_to_f32(MU.stochastic_round_bf16(w, seed=100 + k, step=k))
        errs.append(float(np.mean(out.astype(np.float64) - w.astype(np.float64)) / ulp))
    assert abs(np.mean(errs)) < 1e-3
    # Round to nearest leaves the value unchanged: error is exactly -p ULP.
    rne = MU.bf16_bits_to_f32(MU.f32_to_bf16_rne_bits(w))
    assert np.mean(rne.astype(np.float64) - w) / ulp == pytest.approx(-frac, abs=1e-9)


def test_momentum_closed_form():
    """M_k = G (1 - mu^k) / (1 - mu) for a constant G (Dion3 Eq. 1 with M_0 = 0)."""
    G = np.random.default_rng(2).standard_normal((16, 16)).astype(np.float32)
    mu = 0.95
    M = np.zeros_like(G)
    for _ in range(20):
        M = MU.momentum(M, G, mu)
    np.testing.assert_allclose(M, G * (1 - mu ** 20) / (1 - mu), rtol=1e-5)
    # Exact single step: mu*0 + G == G.
    assert np.array_equal(MU.momentum(np.zeros_like(G), G, mu), G)


def test_update_arithmetic():
    w = np.array([1.0, -2.0, 0.5], np.float32)
    o = np.array([0.25, 0.5, -1.0], np.float32)
    # No decay, unit step: w - o exactly.
    assert np.array_equal(MU.pre_round_update(w, o, 1.0, 0.0, 1.0), w - o)
    # Decay only: (1 - lr*wd) w.
    got = MU.pre_round_update(w, np.zeros(3, np.float32), 0.5, 0.5, 1.0)
    assert np.array_equal(got, np.float32(0.75) * w)
    assert MU.update_scale(4096, 1024) == pytest.approx(0.2 * 64, rel=1e-7)
    assert MU.update_scale(1024, 4096) == MU.update_scale(4096, 1024)


def test_muon_step_matches_definition():
    """One full step on a tiny matrix against the definition written out with
    an SVD-based polar factor replaced by the closed-form NS output."""
    from oracle import gram_ns as O
    rng = np.random.default_rng(3)
    W = MU.f32_to_bf16_rne_bits(0.02 * rng.standard_normal((8, 24)).astype(np.float32))
    G = MU.f32_to_bf16_rne_bits(1e-3 * rng.standard_normal((8, 24)).astype(np.float32))
    M = np.zeros((8, 24), np.float32)
    new_w, new_m, outs = MU.muon_step([W], [G], [M], lr=0.02, wd=0.01, mu=0.95, seed=0, step=2)
    assert np.array_equal(new_m[0], MU.bf16_bits_to_f32(G))
    U, S, Vt = np.linalg.svd(new_m[0].astype(np.float64), full_matrices=False)
    s_hat = S / (1.05 * (np.linalg.norm(new_m[0].astype(np.float64)) + 1e-7))
    o = (U * O.compose_odd_polys(s_hat)) @ Vt
    np.testing.assert_allclose(outs[0], o, rtol=1e-10, atol=1e-12)
    w_new = MU.bf16_bits_to_f32(new_w[0]).astype(np.float64)
    want = (1 - 0.02 * 0.01) * MU.bf16_bits_to_f32(W) - 0.02 * 0.2 * np.sqrt(24) * o
    # Stochastic rounding moves each element by less than one bf16 ULP.
    ulp = np.abs(want) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(w_new - want) <= ulp)


# ---------------------------------------------------------------- NorMuon
# Pins of Dion3 Eq. 2 (NorMuon): the second moment's recursion, the row
# balance it produces, the Frobenius rescale, and its reduction to Muon when
# the rows of O already have equal norms.

def _rows_with_scales(R, C, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((R, C)) * np.exp(rng.uniform(-3, 3, size=(R, 1)))


def test_normuon_second_moment_recursion():
    O = _rows_with_scales(6, 10, 1)
    v0 = np.random.default_rng(2).uniform(0, 1, 6)
    _, v1 = MU.normuon_normalize(O, v0, 0.9, 1e-8)
    want = 0.9 * v0 + 0.1 * np.array([np.dot(r, r) / 10 for r in O])  # mean over the m = 10 columns
    assert np.allclose(v1, want, rtol=1e-14)
    _, vz = MU.normuon_normalize(np.zeros((6, 10)), v0, 0.9, 1e-8)
    assert np.allclose(vz, 0.9 * v0, rtol=1e-15)


def test_normuon_balances_rows_and_keeps_the_frobenius_norm():
    O = _rows_with_scales(8, 24, 3)
    U, _ = MU.normuon_normalize(O, np.zeros(8), 0.0, 0.0)
    # beta2 = 0, eps = 0: v_i is the mean square of row i, so every row of O^
    # has unit RMS and every row of U the same norm ||O|| / sqrt(R).
    row_norms = np.linalg.norm(U, axis=1)
    assert np.allclose(row_norms, np.linalg.norm(O) / np.sqrt(8), rtol=1e-12)
    assert np.isclose(np.linalg.norm(U), np.linalg.norm(O), rtol=1e-14)
    assert np.all(np.sign(U) == np.sign(O))  # a positive scale per row
    # The columns are not balanced (normalizing columns instead would be).
    col_norms = np.linalg.norm(U, axis=0)
    assert col_norms.std() / col_norms.mean() > 1e-2
    # Any beta2 and eps keep the Frobenius norm.
    U2, _ = MU.normuon_normalize(O, np.random.default_rng(4).uniform(0, 2, 8), 0.95, 1e-3)
    assert np.isclose(np.linalg.norm(U2), np.linalg.norm(O), rtol=1e-14)


def test_normuon_equals_muon_for_equal_row_norms():
    """An input with orthonormal rows normalizes to kappa X (all normalized
    singular values equal), so O has equal row norms and NorMuon's direction
    is exactly O: NorMuon reduces to Muon."""
    X = gen.orthonormal_rows_matrix(16, 64, seed=5, dtype=np.float64)
    O = O_NS.orthogonalize(X)
    U, _ = MU.normuon_normalize(O, np.zeros(16), 0.95, 1e-8)
    assert np.allclose(U, O, rtol=1e-12, atol=1e-14)


def test_normuon_step_composes_the_pieces():
    R, C = 12, 40
    w, g = gen.muon_param_inputs(R, C, seed=8, index=0)
    w_bits, g_bits = MU.f32_to_bf16_rne_bits(w), MU.f32_to_bf16_rne_bits(g)
    m0 = np.zeros((R, C), np.float32)
    v0 = np.zeros(R)
    new_w, new_m, new_v, dirs = MU.normuon_step([w_bits], [g_bits], [m0], [v0], 0.02, 0.01, 0.9, 0.95, 1e-8,
                                                seed=1, step=3, base_indices=[77])
    m1 = MU.momentum(m0, MU.bf16_bits_to_f32(g_bits), 0.9)
    U, v1 = MU.normuon_normalize(O_NS.orthogonalize(m1.astype(np.float64)), v0, 0.95, 1e-8)
    assert np.array_equal(new_m[0], m1)
    assert np.allclose(new_v[0], v1) and np.allclose(dirs[0], U)
    want = MU.muon_update_bf16(w_bits, U.astype(np.float32), 0.02, 0.01, MU.update_scale(R, C), 1, 3, 77)
    assert np.array_equal(new_w[0], want)


def test_normuon_eps_outside_the_square_root():
    """Row i of U is O_i / (sqrt(v_i) + eps) times one common factor: with a
    large eps the ratio of two rows' scales pins where eps enters."""
    O = np.array([[3.0, 4.0, 0.0], [0.0, 0.6, 0.8]])
    eps = 0.5
    U, v = MU.normuon_normalize(O, np.zeros(2), 0.0, eps)
    assert np.allclose(v, [25.0 / 3, 1.0 / 3], rtol=1e-15)
    scale = np.linalg.norm(U, axis=1) / np.linalg.norm(O, axis=1)
    want = (np.sqrt(v[1]) + eps) / (np.sqrt(v[0]) + eps)
    assert np.isclose(scale[0] / scale[1], want, rtol=1e-14)


@pytest.mark.parametrize("shape", [(96, 200), (256, 1024)])
def test_sr_update_check_separates_rounding_noise_from_error(shape):
    """The GPU tests judge a stochastically rounded update with
    gpu_helpers.sr_update_error, which subtracts the expected rounding noise.
    Pinned here on the oracle alone: an update computed from an
    orthogonalized matrix with a planted relative error of 0, 2 or 3 % passes
    and its estimated error is the planted one; 4 and 5 % fail."""
    from gpu_helpers import sr_update_error
    r, c = shape
    rng = np.random.default_rng(r * c)
    w = MU.f32_to_bf16_rne_bits((0.02 * rng.standard_normal((r, c))).astype(np.float32))
    o = rng.standard_normal((r, c)) / np.sqrt(max(r, c))
    s = MU.update_scale(r, c)
    for planted, expect in ((0.0, True), (0.02, True), (0.03, True), (0.04, False), (0.05, False)):
        d = rng.standard_normal((r, c))
        d *= planted * np.linalg.norm(o) / np.linalg.norm(d)
        got = MU.muon_update_bf16(w, (o + d).astype(np.float32), 0.02, 0.01, s, seed=7, step=3)
        ok, est, _ = sr_update_error(got, w, o, 0.02, 0.01, s)
        assert ok == expect, (planted, est)
        assert abs(est - planted) < 2e-3, (planted, est)

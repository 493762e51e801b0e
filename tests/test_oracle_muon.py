"""Pins of the Muon elementwise oracle: Philox known answers, the exactness
and unbiasedness of stochastic rounding, and closed forms of the momentum and
update arithmetic."""
import os

import numpy as np
import pytest

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

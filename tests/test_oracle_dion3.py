"""Pins of the Dion3 update rule oracle (Dion3 §6, Algorithm 4, Muon
flavor): the selection, the orthogonalized submatrix, the untouched rows,
the error feedback, and the reduction to Muon at f = 1."""
import numpy as np

from inputs import generators as gen
from oracle import dion3 as D3
from oracle import gram_ns as O_NS
from oracle import muon as MU


def test_selection_count_and_order():
    assert [D3.selection_count(1024, f) for f in (1, 0.5, 0.25, 0.125)] == [1024, 512, 256, 128]
    assert D3.selection_count(10, 0.25) == 3 and D3.selection_count(3, 0.01) == 1
    M = np.array([[1.0, -1.0], [3.0, 0.0], [0.0, -0.5], [2.0, 1.0], [-2.0, 1.0]])
    # l1 norms 2, 3, 0.5, 3, 3: the three 3s first by index, then the 2.
    assert list(D3.select(M, 0.8)) == [1, 3, 4, 0]
    assert list(D3.select(M, 0.4)) == [1, 3]
    # The l1 norm, not the l2 norm: a spread row beats a peaked one.
    P = np.array([[3.0, 0.0, 0.0, 0.0], [1.0, 1.0, 1.0, 1.0], [0.1, 0.0, 0.0, 0.0]])
    assert list(D3.select(P, 0.3)) == [1]


def _inputs(R, C, seed):
    w, g = gen.muon_param_inputs(R, C, seed=seed, index=0)
    m = gen.gaussian(R, C, seed=seed + 1, index=0, scale=1e-3)
    return MU.f32_to_bf16_rne_bits(w), MU.f32_to_bf16_rne_bits(g), m


def test_selected_rows_follow_the_orthogonalized_submatrix():
    R, C, f = 32, 96, 0.25
    w_bits, g_bits, m = _inputs(R, C, 3)
    new_w, new_m, S, O = D3.dion3_step(w_bits, g_bits, m, f, lr=0.02, wd=0.0, mu=0.9, seed=1, step=2)
    M1 = MU.momentum(m, MU.bf16_bits_to_f32(g_bits), 1.0)
    assert np.array_equal(S, D3.select(M1, f)) and len(S) == 8
    assert np.allclose(O, O_NS.orthogonalize(M1[S].astype(np.float64)), rtol=1e-12, atol=1e-15)
    # The selected rows' l1 norms dominate the others'.
    l1 = np.abs(M1.astype(np.float64)).sum(axis=1)
    rest = np.setdiff1d(np.arange(R), S)
    assert l1[S].min() >= l1[rest].max()
    # wd = 0: unselected rows of W are untouched (bf16 values round to themselves).
    assert np.array_equal(new_w[rest], w_bits[rest])
    w0 = MU.bf16_bits_to_f32(w_bits).astype(np.float64)
    delta = MU.bf16_bits_to_f32(new_w).astype(np.float64) - w0
    step = 0.02 * float(MU.update_scale(R, C)) * O
    # One stochastic rounding: within one bf16 ULP of the fp32 result.
    w_new = MU.bf16_bits_to_f32(new_w[S]).astype(np.float64)
    ulp = np.maximum(np.abs(w0[S]), np.abs(w_new)) * 2.0 ** -7
    assert np.all(np.abs(delta[S] + step) <= ulp + 1e-12)


def test_error_feedback_decays_only_the_selected_rows():
    R, C = 24, 64
    w_bits, g_bits, m = _inputs(R, C, 5)
    _, new_m, S, _ = D3.dion3_step(w_bits, g_bits, m, 0.5, lr=0.02, wd=0.01, mu=0.9, seed=1, step=2)
    M1 = MU.momentum(m, MU.bf16_bits_to_f32(g_bits), 1.0)
    rest = np.setdiff1d(np.arange(R), S)
    assert np.array_equal(new_m[rest], M1[rest])
    assert np.array_equal(new_m[S], np.float32(0.9) * M1[S])


def test_weight_decay_applies_to_every_row():
    R, C = 16, 48
    w_bits, g_bits, m = _inputs(R, C, 7)
    new_w, _, S, _ = D3.dion3_step(w_bits, g_bits, m, 0.25, lr=0.1, wd=0.5, mu=0.9, seed=1, step=2)
    rest = np.setdiff1d(np.arange(R), S)
    w0 = MU.bf16_bits_to_f32(w_bits[rest]).astype(np.float64)
    got = MU.bf16_bits_to_f32(new_w[rest]).astype(np.float64)
    assert np.all(np.abs(got - 0.95 * w0) <= np.abs(w0) * 2.0 ** -7 + 1e-12)


def test_columns_are_selected_when_they_are_the_smaller_dimension():
    R, C = 80, 20
    w_bits, g_bits, m = _inputs(R, C, 9)
    new_w, new_m, S, O = D3.dion3_step(w_bits, g_bits, m, 0.25, lr=0.02, wd=0.0, mu=0.9, seed=1, step=2)
    M1 = MU.momentum(m, MU.bf16_bits_to_f32(g_bits), 1.0)
    assert np.array_equal(S, D3.select(M1.T, 0.25)) and O.shape == (5, R)
    rest = np.setdiff1d(np.arange(C), S)
    assert np.array_equal(new_w[:, rest], w_bits[:, rest])
    assert np.array_equal(new_m[:, S], np.float32(0.9) * M1[:, S])


def test_full_fraction_reduces_to_muon():
    """f = 1 selects every row; the update equals Muon's on the same momentum
    (rows permuted by the selection, then put back)."""
    R, C = 24, 80
    w_bits, g_bits, m = _inputs(R, C, 11)
    new_w, _, S, O = D3.dion3_step(w_bits, g_bits, m, 1.0, lr=0.02, wd=0.01, mu=0.9, seed=1, step=2)
    M1 = MU.momentum(m, MU.bf16_bits_to_f32(g_bits), 1.0)
    O_muon = O_NS.orthogonalize(M1.astype(np.float64))
    back = np.zeros_like(O_muon)
    back[S] = O
    assert np.allclose(back, O_muon, rtol=1e-10, atol=1e-13)
    want = MU.muon_update_bf16(w_bits, back.astype(np.float32), 0.02, 0.01, MU.update_scale(R, C), 1, 2, 0)
    assert np.array_equal(new_w, want)

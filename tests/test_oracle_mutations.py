"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake (a dropped term, a wrong sign, a swapped
operand or coefficient, a misplaced restart, a lost transpose or safety
factor) into a private copy of the oracle's source, on the CPU, and checks
that at least one pin fails for the mutant while all pass for the original.
"""
import importlib.util
import os
import sys

import numpy as np
import pytest

from inputs import generators as gen

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "gram_ns.py")

MUTANTS = {
    "drop_aR_in_RZ": ("RZ = _mm(counter, R, Z, symmetric=True) + a * R",
                      "RZ = _mm(counter, R, Z, symmetric=True)"),
    "sign_aRZ": ("R = _mm(counter, Z, RZ, symmetric=True) + a * RZ",
                 "R = _mm(counter, Z, RZ, symmetric=True) - a * RZ"),
    "drop_aI_at_reset": ("Q = Z + a * I\n", "Q = Z\n"),
    "wrong_operand_in_Q": ("Q = _mm(counter, Q, Z, symmetric=True) + a * Q",
                           "Q = _mm(counter, Q, Z, symmetric=True) + a * Z"),
    "swap_b_c": ("Z = b * R + c * _mm(counter, R, R, symmetric=True)",
                 "Z = c * R + b * _mm(counter, R, R, symmetric=True)"),
    "restart_one_late": ("if (t - 1) in restarts:", "if (t - 2) in restarts:"),
    "no_safety_factor": ('return X / (SAFETY * (np.linalg.norm(X, "fro") + EPS))',
                         'return X / (np.linalg.norm(X, "fro") + EPS)'),
    "transposed_gram": ("    R = _mm(counter, X, X.T, symmetric=True)\n    Q = None  # identity; the first",
                        "    R = _mm(counter, X.T, X, symmetric=True)[:X.shape[0], :X.shape[0]]\n    Q = None  # identity; the first"),
    "restart_uses_old_Q_transposed": ("            X = _mm(counter, Q, X)\n",
                                      "            X = _mm(counter, Q.T @ Q, X)\n"),
    "std_ns_drop_aX": ("X = a * X + _mm(counter, B, X)", "X = _mm(counter, B, X)"),
    "naive_R_update_order": ("R = _mm(counter, ZR, Z, symmetric=True)",
                             "R = _mm(counter, ZR, ZR, symmetric=True)"),
    "lost_back_transpose": ("    out = _mm(counter, Q, X)\n    return out.T if transposed else out\n\n\ndef orthogonalize(",
                            "    out = _mm(counter, Q, X)\n    return out\n\n\ndef orthogonalize("),
    "skip_R_update_always": ("if t < steps and t not in restarts:", "if t < steps - 1 and t not in restarts:"),
}


def load_variant(name, source):
    spec = importlib.util.spec_from_loader(name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(source, name, "exec"), mod.__dict__)
    return mod


def closed_form(X, O):
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    s_hat = S / (1.05 * (np.linalg.norm(X) + 1e-7))
    p = s_hat.copy()
    for _ in range(5):
        a, b, c = 3.4445, -4.7750, 2.0315
        p = a * p + b * p ** 3 + c * p ** 5
    return (U * p) @ Vt


def pins_pass(O):
    """A battery of the oracle pins; True when every one holds."""
    try:
        for shape in ((8, 32), (24, 10), (6, 6)):
            X = gen.gaussian(*shape, seed=31).astype(np.float64)
            want = closed_form(X, O)
            for out in (O.gram_ns(X), O.standard_ns(X), O.gram_ns_naive(X), O.orthogonalize(X)):
                if out.shape != want.shape:
                    return False
                if np.linalg.norm(out - want) > 1e-10 * np.linalg.norm(want):
                    return False
        trace = []
        O.gram_ns(gen.gaussian(8, 24, seed=1).astype(np.float64), trace=trace)
        seq = [(t, n) for t, n, _ in trace]
        if seq != [(0, "R"), (1, "Z"), (1, "Q"), (1, "RZ"), (1, "R"), (2, "Z"), (2, "Q"),
                   (3, "X"), (3, "R"), (3, "Z"), (3, "Q"), (3, "RZ"), (3, "R"),
                   (4, "Z"), (4, "Q"), (4, "RZ"), (4, "R"), (5, "Z"), (5, "Q")]:
            return False
        n, m = 16, 64
        c = O.FlopCounter()
        O.gram_ns(gen.gaussian(n, m, seed=2).astype(np.float64), counter=c)
        if c.flops != (4 * 5 + 6 * 4 - 6) * n ** 3:
            return False
    except Exception:
        return False
    return True


def test_original_passes():
    assert pins_pass(load_variant("oracle_original", open(SRC).read()))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site not unique/found: {name}"
    assert not pins_pass(load_variant(f"oracle_{name}", src.replace(old, new)))


# NorMuon (Dion3 Eq. 2) in oracle/muon.py: the same check against its pins.
MU_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "muon.py")

NORMUON_MUTANTS = {
    "normuon_mean_over_rows": ("np.sum(O * O, axis=1) / m", "np.sum(O * O, axis=1) / O.shape[0]"),
    "normuon_drop_one_minus_beta2": ("(1.0 - beta2) * np.sum(O * O, axis=1)", "np.sum(O * O, axis=1)"),
    "normuon_eps_inside_sqrt": ("(np.sqrt(v_new) + eps)", "np.sqrt(v_new + eps)"),
    "normuon_no_rescale": ("U = O_hat * (n_o / n_hat) if n_hat > 0", "U = O_hat if n_hat > 0"),
    "normuon_rescale_inverted": ("U = O_hat * (n_o / n_hat) if n_hat > 0", "U = O_hat * (n_hat / n_o) if n_hat > 0"),
    "normuon_columns": ("O_hat = O / (np.sqrt(v_new) + eps)[:, None]",
                        "O_hat = (O.T / (np.sqrt(v_new) + eps)[: O.shape[1], None]).T"),
}


def normuon_pins_pass(MU):
    import tests.test_oracle_muon as T
    saved = T.MU
    T.MU = MU
    try:
        for fn in (T.test_normuon_second_moment_recursion, T.test_normuon_balances_rows_and_keeps_the_frobenius_norm,
                   T.test_normuon_equals_muon_for_equal_row_norms, T.test_normuon_eps_outside_the_square_root):
            fn()
    except Exception:
        return False
    finally:
        T.MU = saved
    return True


def test_normuon_original_passes():
    assert normuon_pins_pass(load_variant("muon_original", open(MU_SRC).read()))


@pytest.mark.parametrize("name", sorted(NORMUON_MUTANTS))
def test_normuon_mutant_is_caught(name):
    src = open(MU_SRC).read()
    old, new = NORMUON_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site not unique/found: {name}"
    assert not normuon_pins_pass(load_variant(f"muon_{name}", src.replace(old, new)))


# Dion3 update rule (Algorithm 4) in oracle/dion3.py.
D3_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "dion3.py")

DION3_MUTANTS = {
    "dion3_smallest_rows": ("order = np.lexsort((np.arange(n), -l1))", "order = np.lexsort((np.arange(n), l1))"),
    "dion3_l2_selection": ("l1 = np.abs(M).sum(axis=1)", "l1 = (M * M).sum(axis=1)"),
    "dion3_damp_every_row": ("        M_new[S] = np.float32(mu) * M_new[S]", "        M_new = np.float32(mu) * M_new"),
    "dion3_momentum_damped_first": ("M = MU.momentum(M, MU.bf16_bits_to_f32(g_bits), 1.0)",
                                    "M = MU.momentum(M, MU.bf16_bits_to_f32(g_bits), mu)"),
    "dion3_rows_always": ("cols = R > C", "cols = False"),
    "dion3_floor_count": ("int(math.ceil(f * n - 1e-9))", "int(math.floor(f * n))"),
}


def dion3_pins_pass(D3):
    import tests.test_oracle_dion3 as T
    saved = T.D3
    T.D3 = D3
    try:
        for name in dir(T):
            if name.startswith("test_"):
                getattr(T, name)()
    except Exception:
        return False
    finally:
        T.D3 = saved
    return True


def load_oracle_module(name, source):
    spec = importlib.util.spec_from_loader(f"oracle.{name}", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(source, name, "exec"), mod.__dict__)
    return mod


def test_dion3_original_passes():
    assert dion3_pins_pass(load_oracle_module("dion3_original", open(D3_SRC).read()))


@pytest.mark.parametrize("name", sorted(DION3_MUTANTS))
def test_dion3_mutant_is_caught(name):
    src = open(D3_SRC).read()
    old, new = DION3_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site not unique/found: {name}"
    assert not dion3_pins_pass(load_oracle_module(f"dion3_{name}", src.replace(old, new)))

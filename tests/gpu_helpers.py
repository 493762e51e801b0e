"""Helpers shared by the GPU tests: parity metrics against the oracle."""
import numpy as np

# Tolerances of the parity bar: per matrix, relative Frobenius error <= 3e-2,
# cosine >= 0.98, max singular-value deviation <= 0.05, no NaN/Inf.
REL_TOL = 3e-2
COS_TOL = 0.98
SV_TOL = 0.05


def parity_metrics(got, ref, with_sv=True):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    finite = bool(np.all(np.isfinite(got)))
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nref if nref > 0 else np.linalg.norm(got)
    denom = np.linalg.norm(got) * nref
    cos = float(np.sum(got * ref) / denom) if denom > 0 else (1.0 if np.linalg.norm(got) == 0 else 0.0)
    sv = 0.0
    if with_sv and finite:
        s_got = np.linalg.svd(got, compute_uv=False)
        s_ref = np.linalg.svd(ref, compute_uv=False)
        sv = float(np.max(np.abs(np.sort(s_got) - np.sort(s_ref))))
    return dict(finite=finite, rel=float(rel), cos=cos, sv=sv)


def assert_parity(got, ref, with_sv=True, what=""):
    m = parity_metrics(got, ref, with_sv)
    assert m["finite"], f"{what}: non-finite output"
    assert m["rel"] <= REL_TOL, f"{what}: relative error {m['rel']:.3e}"
    assert m["cos"] >= COS_TOL, f"{what}: cosine {m['cos']:.5f}"
    assert m["sv"] <= SV_TOL, f"{what}: singular-value deviation {m['sv']:.3e}"
    return m

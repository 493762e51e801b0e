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


def sr_update_error(got_bits, w_old_bits, o_ref, lr, wd, scale, tol=REL_TOL, sigmas=4.0):
    """Parity of a stochastically rounded weight update against the oracle.

    got = SR(w'_gpu) with w'_gpu = (1 - lr wd) w - lr s o_gpu. Against the
    oracle's unrounded w'_ref (the same formula with the oracle's o):
    got - w'_ref = delta + e, where delta = w'_gpu - w'_ref is the
    orthogonalization's error times lr s, and e is the rounding error of one
    stochastic rounding: zero mean, and for an element whose fraction between
    its two bf16 neighbours (ULP apart) is p, e^2 has mean p (1 - p) ULP^2.
    So ||got - w'_ref||^2 - sum p (1 - p) ULP^2 estimates ||delta||^2 without
    the rounding noise. The check passes when that estimate is at most
    (tol ||lr s o_ref||)^2 plus `sigmas` standard deviations of the noise
    terms (the spread of sum e^2 and of the cross term 2 <delta, e> with
    |delta| at the bar). Returns (ok, estimated relative error, details)."""
    from oracle import muon as MU
    w_old = MU.bf16_bits_to_f32(w_old_bits)
    o32 = np.asarray(o_ref, np.float64).astype(np.float32)
    w_pre = MU.pre_round_update(w_old, o32, lr, wd, scale)
    got = MU.bf16_bits_to_f32(got_bits).astype(np.float64)
    assert np.all(np.isfinite(got)), "non-finite weights"
    bits = w_pre.view(np.uint32).astype(np.uint64)
    trunc = bits & np.uint64(0xFFFF0000)
    lo = (trunc.astype(np.uint32)).view(np.float32).astype(np.float64)
    hi = ((trunc + np.uint64(0x10000)).astype(np.uint32)).view(np.float32).astype(np.float64)
    ulp = np.abs(hi - lo)
    p = (bits & np.uint64(0xFFFF)).astype(np.float64) / 65536.0
    q = p * (1.0 - p)
    upd = np.float64(np.float32(lr) * np.float32(scale)) * o32.astype(np.float64)
    n_upd = np.linalg.norm(upd)
    d2 = float(np.sum((got - w_pre.astype(np.float64)) ** 2))
    v = float(np.sum(q * ulp ** 2))
    var_e2 = float(np.sum(q * ((1 - p) ** 2 + p ** 2) * ulp ** 4 - (q * ulp ** 2) ** 2))
    var_cross = float(4.0 * np.sum((tol * upd) ** 2 * q * ulp ** 2))
    sigma = np.sqrt(var_e2 + var_cross)
    est = np.sqrt(max(d2 - v, 0.0)) / n_upd
    ok = d2 - v <= (tol * n_upd) ** 2 + sigmas * sigma
    return bool(ok), float(est), dict(d2=d2, noise=v, sigma=float(sigma), upd=float(n_upd))

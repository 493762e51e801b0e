"""CPU oracle for the Muon elementwise steps around the orthogonalization.

TEST INFRASTRUCTURE ONLY (same rule as ``oracle/gram_ns.py``: only tests/,
``__graft_entry__.smoke()`` and bench.py's CPU legs use it).

What it computes:

* Momentum: M <- mu M + G with M_0 = 0 ("Dion3: Full-stack orthogonal
  updates", §2.1, Eq. 1). fp32, each operation rounded once (no fused
  multiply-add), G promoted from bf16.
* Update: W <- (1 - lr*wd) W - lr*s*O, decoupled weight decay and the scaled
  update in one pass, in fp32 with one final downcast (Dion3 §6 "Weight
  Update", Algorithm 4 weight-decay and update lines; the grouped Muon kernel
  card, "How it works"). Operation order, each rounded to nearest fp32:
  decay = 1 - lr*wd; step = lr*s; w' = decay*w - step*o.
* Scale s = 0.2 * sqrt(max(rows, cols)): the Moonshot rule that Dion3 App. A.1
  reports as the best for its Muon runs.
* NorMuon flavor (Dion3 §2.1, Eq. 2): after O = polar(M), per row i of the
  weight's shape, v_i <- beta2 v_i + (1 - beta2) (1/m) sum_j O_ij^2 with m the
  number of columns; O^_ij = O_ij / (sqrt(v_i) + eps); the update direction is
  O^ rescaled to the Frobenius norm of O. Readings: the same decoupled weight
  decay and scale s as the Muon flavor apply on top (Dion3 §6 applies weight
  decay before either flavor's update); v starts at zero and is the caller's
  state like M. Computed in fp64 here (Dion3 §6 asks for at least fp32).
* Stochastic rounding of w' to bf16, keyed by the element's global index
  (the grouped Muon kernel card: "counter-based stochastic rounding keyed by
  the element's global index", "base_index sets the global-index offset").
  The card names no generator. Reading: Philox4x32-10 (Salmon, Moraes, Dror,
  Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11). For global
  index g = base_index + i, counter = (g >> 3 as two 32-bit words, step as two
  32-bit words), key = (seed low word, seed high word); one output (four
  32-bit words) serves the eight elements of a block: element g takes the
  16-bit half (g & 1) (low half first) of output word (g & 7) >> 1.
  bf16 = high 16 bits of (bits(w') + u). NaN stays NaN (quiet bit set);
  +-Inf stays as is.
"""
from __future__ import annotations

import numpy as np

PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint32(0x9E3779B9)
PHILOX_W1 = np.uint32(0xBB67AE85)
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds (Salmon et al., SC'11, §4.2 and Table 2).

    Each round: (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2 (64-bit products),
    new counter = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); the key is bumped
    by the Weyl constants (W0, W1) between rounds. Arrays of uint32 in,
    four uint32 arrays out."""
    c0 = np.asarray(c0, dtype=np.uint32).astype(np.uint64)
    c1 = np.asarray(c1, dtype=np.uint32).astype(np.uint64)
    c2 = np.asarray(c2, dtype=np.uint32).astype(np.uint64)
    c3 = np.asarray(c3, dtype=np.uint32).astype(np.uint64)
    k0 = np.uint64(np.uint32(k0))
    k1 = np.uint64(np.uint32(k1))
    for r in range(10):
        if r > 0:
            k0 = (k0 + np.uint64(PHILOX_W0)) & MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & MASK32
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return tuple(v.astype(np.uint32) for v in (c0, c1, c2, c3))


def sr_uniform16(global_index, seed, step):
    """The 16-bit random value each element adds before truncation."""
    g = np.asarray(global_index, dtype=np.uint64)
    blk = g >> np.uint64(3)
    lane = ((g & np.uint64(7)) >> np.uint64(1)).astype(np.int64)
    half = (g & np.uint64(1)).astype(np.uint32)
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    step = int(step) & 0xFFFFFFFFFFFFFFFF
    outs = philox4x32_10(blk & MASK32, blk >> np.uint64(32),
                         np.full(blk.shape, step & 0xFFFFFFFF, dtype=np.uint32),
                         np.full(blk.shape, step >> 32, dtype=np.uint32),
                         seed & 0xFFFFFFFF, seed >> 32)
    stacked = np.stack(outs, axis=-1)
    word = np.take_along_axis(stacked, lane[..., None], axis=-1)[..., 0]
    return ((word >> (np.uint32(16) * half)) & np.uint32(0xFFFF)).astype(np.uint32)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_rne_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bits (for building inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    r = np.where(nan, (b >> np.uint64(16)) | np.uint64(0x40), r)
    return r.astype(np.uint16)


def stochastic_round_bf16(w, seed, step, base_index=0):
    """bf16 bits of w (fp32 array, row-major) rounded stochastically."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    bits = w.view(np.uint32).astype(np.uint64)
    idx = np.arange(w.size, dtype=np.uint64).reshape(w.shape) + np.uint64(base_index)
    u = sr_uniform16(idx, seed, step).astype(np.uint64)
    rounded = (bits + u) >> np.uint64(16)
    finite = np.isfinite(w)
    nan = np.isnan(w)
    out = np.where(finite, rounded, bits >> np.uint64(16))
    out = np.where(nan, (bits >> np.uint64(16)) | np.uint64(0x40), out)
    return out.astype(np.uint16)


def momentum(M, G, mu):
    """M <- mu M + G in fp32, two roundings (Dion3 Eq. 1)."""
    M = np.asarray(M, dtype=np.float32)
    G = np.asarray(G, dtype=np.float32)
    return np.float32(mu) * M + G


def update_scale(rows, cols):
    """0.2 * sqrt(max(fan_out, fan_in)) in fp32 (Dion3 App. A.1)."""
    return np.float32(0.2) * np.sqrt(np.float32(max(rows, cols)))


def pre_round_update(w, o, lr, wd, scale):
    """w' = (1 - lr*wd) w - (lr*s) o in fp32, each operation rounded once."""
    w = np.asarray(w, dtype=np.float32)
    o = np.asarray(o, dtype=np.float32)
    decay = np.float32(1.0) - np.float32(lr) * np.float32(wd)
    stepv = np.float32(lr) * np.float32(scale)
    return decay * w - stepv * o


def muon_update_bf16(w_bits, o, lr, wd, scale, seed, step, base_index=0):
    """One fused update of a bf16 weight matrix (bits in, bits out)."""
    w = bf16_bits_to_f32(w_bits)
    w_new = pre_round_update(w, o, lr, wd, scale)
    return stochastic_round_bf16(w_new, seed, step, base_index)


def muon_step(params_bits, grads_bits, momenta, lr, wd, mu, seed, step,
              base_indices=None, ns=None):
    """A full Muon step over a list of matrices (Dion3 Eq. 1 with decoupled
    weight decay). ``ns`` maps an fp32 matrix to its orthogonalized fp64
    matrix (defaults to the Gram NS oracle). Returns (new param bits, new
    momenta, orthogonalized matrices)."""
    from .gram_ns import orthogonalize
    ns = ns or orthogonalize
    if base_indices is None:
        base_indices = [0] * len(params_bits)
    new_w, new_m, outs = [], [], []
    for w_bits, g_bits, m, base in zip(params_bits, grads_bits, momenta, base_indices):
        m_new = momentum(m, bf16_bits_to_f32(g_bits), mu)
        o = ns(m_new.astype(np.float64))
        s = update_scale(*w_bits.shape)
        new_w.append(muon_update_bf16(w_bits, o.astype(np.float32), lr, wd, s, seed, step, base))
        new_m.append(m_new)
        outs.append(o)
    return new_w, new_m, outs


def normuon_normalize(O, v, beta2, eps):
    """NorMuon's steps after the orthogonalization (Dion3 Eq. 2), in fp64:
    returns (U, v_new) with v_new_i = beta2 v_i + (1 - beta2) mean_j O_ij^2,
    O^ = O / (sqrt(v_new) + eps) row by row, and U = (||O||_F / ||O^||_F) O^
    (zero when O^ is zero)."""
    O = np.asarray(O, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m = O.shape[1]
    v_new = beta2 * v + (1.0 - beta2) * np.sum(O * O, axis=1) / m
    O_hat = O / (np.sqrt(v_new) + eps)[:, None]
    n_o, n_hat = np.linalg.norm(O), np.linalg.norm(O_hat)
    U = O_hat * (n_o / n_hat) if n_hat > 0 else np.zeros_like(O_hat)
    return U, v_new


def normuon_step(params_bits, grads_bits, momenta, second_moments, lr, wd, mu, beta2, eps, seed, step,
                 base_indices=None, ns=None):
    """A full NorMuon step over a list of matrices (Dion3 Eq. 2 with the Muon
    flavor's decoupled weight decay, scale and stochastic rounding). Returns
    (new param bits, new momenta, new second moments, update directions U)."""
    from .gram_ns import orthogonalize
    ns = ns or orthogonalize
    if base_indices is None:
        base_indices = [0] * len(params_bits)
    new_w, new_m, new_v, dirs = [], [], [], []
    for w_bits, g_bits, m, v, base in zip(params_bits, grads_bits, momenta, second_moments, base_indices):
        m_new = momentum(m, bf16_bits_to_f32(g_bits), mu)
        U, v_new = normuon_normalize(ns(m_new.astype(np.float64)), v, beta2, eps)
        s = update_scale(*w_bits.shape)
        new_w.append(muon_update_bf16(w_bits, U.astype(np.float32), lr, wd, s, seed, step, base))
        new_m.append(m_new)
        new_v.append(v_new)
        dirs.append(U)
    return new_w, new_m, new_v, dirs

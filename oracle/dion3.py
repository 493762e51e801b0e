"""CPU oracle for the Dion3 update rule ("Dion3: Full-stack orthogonal
updates", §6 and Algorithm 4), Muon flavor.

TEST INFRASTRUCTURE ONLY (same rule as ``oracle/gram_ns.py``: only tests/,
``__graft_entry__.smoke()`` and bench.py's CPU legs use it).

One weight matrix W (rows x cols), gradient G, momentum M, fraction f:

1. M <- M + G (fp32, one rounding; Algorithm 4 accumulates before damping).
2. Selection along the smaller dimension (§6 "Selection": with no sharding,
   whichever dimension is smaller; rows on a tie): the k = ceil(f n) rows
   (or columns) of M with the largest l1 norm. Reading: equal norms are
   ordered by index, lower first; the selected rows keep that order
   (largest norm first) in the submatrix.
3. O = polar(M[S, :]), here the Gram Newton-Schulz oracle (5 quintic steps,
   one restart), which the GPU path uses too.
4. W <- (1 - lr wd) W for every row; W[S, :] <- ... - lr s O for the selected
   rows, as one fp32 operation per element followed by the stochastic
   rounding of the Muon flavor (§6 "Weight Update": decay applied to all
   rows, then the selected rows updated; one fused fp32 pass). Reading: s =
   0.2 sqrt(max(rows, cols)) of the whole parameter, as for Muon.
5. Error feedback: M[S, :] <- mu M[S, :] (fp32), other rows unchanged
   (§6 "Error Feedback").
"""
from __future__ import annotations

import math

import numpy as np

from . import muon as MU


def selection_count(n, f):
    """k = ceil(f n), at least 1 and at most n."""
    return max(1, min(n, int(math.ceil(f * n - 1e-9))))


def select(M, f):
    """Indices of the k rows of M with the largest l1 norm, largest first,
    equal norms by lower index (fp64 norms)."""
    M = np.asarray(M, dtype=np.float64)
    n = M.shape[0]
    l1 = np.abs(M).sum(axis=1)
    order = np.lexsort((np.arange(n), -l1))
    return order[:selection_count(n, f)]


def dion3_step(w_bits, g_bits, M, f, lr, wd, mu, seed, step, base_index=0, ns=None):
    """One Dion3 step (Muon flavor) for one matrix. Returns (new W bits, new M,
    selected indices along the selection dimension, O)."""
    from .gram_ns import orthogonalize
    ns = ns or orthogonalize
    R, C = w_bits.shape
    M = MU.momentum(M, MU.bf16_bits_to_f32(g_bits), 1.0)  # M + G, one rounding
    cols = R > C  # select columns when they are the smaller dimension
    Ms = M.T if cols else M
    S = select(Ms, f)
    O = ns(Ms[S].astype(np.float64))
    full = np.zeros(Ms.shape, dtype=np.float32)
    full[S] = O.astype(np.float32)
    if cols:
        full = full.T
    s = MU.update_scale(R, C)
    new_w = MU.muon_update_bf16(w_bits, full, lr, wd, s, seed, step, base_index)
    M_new = M.copy()
    if cols:
        M_new[:, S] = np.float32(mu) * M_new[:, S]
    else:
        M_new[S] = np.float32(mu) * M_new[S]
    return new_w, M_new, S, O

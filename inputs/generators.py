"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no arithmetic of the method: only random matrices. Both the
oracle-side tests and the GPU side draw their inputs from here, so the two
see identical data. Every matrix is drawn from its own generator seeded by
(seed, index), so matrix g of a bucket does not depend on the bucket size.

Workloads (Dion3 paper and the grouped Muon kernel card):
* MLP-like rectangular buckets, alpha = 4 (Dion3 §4.1 footnote on the 4x
  MLP ratio).
* Square attention projections with singular values log-uniform in
  [1e-6, 1] and Haar-random singular vectors (the card's "ill-conditioned to
  1e-6" class).
* A fine-grained MoE bucket split over the card's conditioning classes:
  Gaussian, low-rank, heavy-tailed, near-orthogonal, scaled by 1e-3 and 1e+3.
* A 7B Llama-like layer stack for the full Muon step (Dion3 Fig. 1 workload).
* A 128 x 512 matrix with an exponentially decaying spectrum (Dion3 App. B.1).
"""
from __future__ import annotations

import numpy as np


def rng_for(seed, index=0):
    return np.random.default_rng([int(seed), int(index)])


def gaussian(rows, cols, seed, index=0, scale=1.0, dtype=np.float32):
    g = rng_for(seed, index).standard_normal((rows, cols))
    return (scale * g).astype(dtype)


def student_t(rows, cols, seed, index=0, nu=3.0, dtype=np.float32):
    return rng_for(seed, index).standard_t(nu, size=(rows, cols)).astype(dtype)


def low_rank(rows, cols, seed, index=0, rank=32, dtype=np.float32):
    r = rng_for(seed, index)
    a = r.standard_normal((rows, rank))
    b = r.standard_normal((rank, cols))
    return (a @ b).astype(dtype)


def haar_orthogonal(n, rng):
    """Haar-distributed orthogonal n x n matrix: QR of a Gaussian matrix with
    the signs of R's diagonal moved into Q (Mezzadri's recipe)."""
    q, r = np.linalg.qr(rng.standard_normal((n, n)))
    d = np.sign(np.diag(r))
    d[d == 0] = 1.0
    return q * d


def orthonormal_rows(rows, cols, rng):
    """rows x cols (rows <= cols) with orthonormal rows."""
    q, r = np.linalg.qr(rng.standard_normal((cols, rows)))
    d = np.sign(np.diag(r))
    d[d == 0] = 1.0
    return (q * d).T


def log_uniform_spectrum(n, seed, index=0, lo=1e-6, hi=1.0, dtype=np.float32):
    """U diag(s) V^T with Haar U, V and s log-uniform in [lo, hi], in fp64."""
    r = rng_for(seed, index)
    u = haar_orthogonal(n, r)
    v = haar_orthogonal(n, r)
    s = np.exp(r.uniform(np.log(lo), np.log(hi), size=n))
    return ((u * s) @ v.T).astype(dtype)


def near_orthogonal(rows, cols, seed, index=0, noise=1e-3, dtype=np.float32):
    """Orthonormal rows plus noise * N(0, 1)."""
    r = rng_for(seed, index)
    q = orthonormal_rows(rows, cols, r)
    return (q + noise * r.standard_normal((rows, cols))).astype(dtype)


def exp_decay_spectrum(rows, cols, seed, index=0, decay=0.1, dtype=np.float64):
    """rows x cols with singular values exp(-decay * i) and random singular
    vectors (the 128 x 512 test matrix of Dion3 App. B.1)."""
    r = rng_for(seed, index)
    n = min(rows, cols)
    u = orthonormal_rows(n, rows, r).T
    v = orthonormal_rows(n, cols, r).T
    s = np.exp(-decay * np.arange(n))
    return ((u * s) @ v.T).astype(dtype)


def orthonormal_rows_matrix(rows, cols, seed, index=0, dtype=np.float32):
    r = rng_for(seed, index)
    if rows <= cols:
        return orthonormal_rows(rows, cols, r).astype(dtype)
    return orthonormal_rows(cols, rows, r).T.astype(dtype)


# ---------------------------------------------------------------------------
# Buckets
# ---------------------------------------------------------------------------

MOE_CLASSES = ("gaussian", "low_rank", "student_t", "near_orthogonal",
               "scaled_1e-3", "scaled_1e+3")


def moe_class_counts(total, classes=MOE_CLASSES):
    """Split ``total`` as evenly as possible over the classes, earlier classes
    taking the remainder (256 over 6 gives 43, 43, 43, 43, 42, 42)."""
    base, extra = divmod(total, len(classes))
    return [base + (1 if i < extra else 0) for i in range(len(classes))]


def moe_class_of(index, total, classes=MOE_CLASSES):
    counts = moe_class_counts(total, classes)
    acc = 0
    for name, c in zip(classes, counts):
        acc += c
        if index < acc:
            return name
    raise IndexError(index)


def moe_matrix(kind, rows, cols, seed, index):
    if kind == "gaussian":
        return gaussian(rows, cols, seed, index)
    if kind == "low_rank":
        return low_rank(rows, cols, seed, index)
    if kind == "student_t":
        return student_t(rows, cols, seed, index)
    if kind == "near_orthogonal":
        return near_orthogonal(rows, cols, seed, index)
    if kind == "scaled_1e-3":
        return gaussian(rows, cols, seed, index, scale=1e-3)
    if kind == "scaled_1e+3":
        return gaussian(rows, cols, seed, index, scale=1e3)
    raise ValueError(kind)


def gaussian_bucket(G, rows, cols, seed, first=0):
    """Matrices first .. first + G - 1 of the seeded Gaussian bucket (each
    from its own (seed, index) generator, so any chunk of a bucket is the
    same data as in the whole bucket)."""
    out = np.empty((G, rows, cols), dtype=np.float32)
    for g in range(G):
        out[g] = gaussian(rows, cols, seed, first + g)
    return out


def conditioned_square_bucket(G, n, seed, lo=1e-6, hi=1.0):
    out = np.empty((G, n, n), dtype=np.float32)
    for g in range(G):
        out[g] = log_uniform_spectrum(n, seed, g, lo, hi)
    return out


def moe_bucket(G, rows, cols, seed):
    out = np.empty((G, rows, cols), dtype=np.float32)
    for g in range(G):
        out[g] = moe_matrix(moe_class_of(g, G), rows, cols, seed, g)
    return out


# Named configurations (seed = 1000 * config number + replica).
CONFIGS = {
    "single_128x512": dict(G=1, rows=128, cols=512, seed=1000),
    "mlp_24x1024x4096": dict(G=24, rows=1024, cols=4096, seed=2000),
    "square_16x2048": dict(G=16, rows=2048, cols=2048, seed=3000),
    "moe_256x512x2048": dict(G=256, rows=512, cols=2048, seed=4000),
}


def config_bucket(name, G=None, replica=0):
    cfg = CONFIGS[name]
    G = cfg["G"] if G is None else G
    seed = cfg["seed"] + replica
    if name == "square_16x2048":
        return conditioned_square_bucket(G, cfg["rows"], seed)
    if name == "moe_256x512x2048":
        return moe_bucket(G, cfg["rows"], cfg["cols"], seed)
    return gaussian_bucket(G, cfg["rows"], cfg["cols"], seed)


# 7B Llama-like stack: per layer q, o (4096^2), k, v (1024 x 4096),
# gate, up (14336 x 4096), down (4096 x 14336); 32 layers.
LLAMA7B_LAYER = (("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096),
                 ("o", 4096, 4096), ("gate", 14336, 4096), ("up", 14336, 4096),
                 ("down", 4096, 14336))
LLAMA7B_LAYERS = 32


def llama7b_shapes(layers=LLAMA7B_LAYERS):
    return [(f"layer{l}.{name}", r, c) for l in range(layers) for name, r, c in LLAMA7B_LAYER]


def muon_param_inputs(rows, cols, seed, index, w_std=0.02, g_std=1e-3):
    """(W fp32 values, G fp32 values) to be rounded to bf16 by the caller:
    W ~ N(0, w_std), G ~ N(0, g_std)."""
    r = rng_for(seed, index)
    w = (w_std * r.standard_normal((rows, cols))).astype(np.float32)
    g = (g_std * r.standard_normal((rows, cols))).astype(np.float32)
    return w, g

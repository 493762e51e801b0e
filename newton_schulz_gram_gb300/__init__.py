"""GB300-native Gram Newton-Schulz orthogonalization and Muon step.

Thin Python binding over libgns.so (include/gns.h): each function marshals
torch tensors into pointers, sizes and the current CUDA stream and calls the
C entry point of the same name. All arithmetic runs in the library's sm_103a
kernels; PyTorch only provides device memory and streams.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import GnsError, GnsTensor, check, load

__all__ = ["gns_orthogonalize_batched", "gns_orthogonalize_batched_host",
           "gns_orthogonalize_batched_noalloc", "gns_orthogonalize_batched_schedule", "muon_step", "normuon_step", "dion3_step",
           "gns_muon_momentum", "gns_muon_update", "gns_symm_gemm", "gns_get_status",
           "gns_status_string", "gns_last_error", "gns_workspace_bytes", "gns_release",
           "gns_launch_count", "gns_profile_enable", "gns_profile_read", "KERNEL_CLASSES",
           "GnsError", "QUINTIC", "load"]

QUINTIC = (3.4445, -4.7750, 2.0315)


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _coeff_array(coeffs, steps):
    if coeffs is None:
        return None, None
    flat = [float(v) for row in coeffs for v in (row if hasattr(row, "__len__") else [row])]
    if len(flat) == 3:
        flat = flat * steps
    if len(flat) != 3 * steps:
        raise ValueError("coeffs must hold 3 or 3*steps values")
    arr = (ctypes.c_float * len(flat))(*flat)
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def _require(t, dtype, cuda=True, name="tensor"):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gns_orthogonalize_batched(x, steps=5, restart_at=2, coeffs=None, stream=None):
    """Orthogonalize x in place: fp32 CUDA tensor [R, C] or [G, R, C]."""
    _require(x, torch.float32, name="x")
    G, R, C = (1, *x.shape) if x.dim() == 2 else tuple(x.shape)
    keep, cptr = _coeff_array(coeffs, steps)
    lib = load()
    check(lib.gns_orthogonalize_batched(ctypes.c_void_p(x.data_ptr()), G, R, C, steps, restart_at,
                                        cptr, _stream(stream, x.device)), "gns_orthogonalize_batched")
    del keep
    return x


def gns_orthogonalize_batched_schedule(x, steps=5, restarts=(2,), coeffs=None, stream=None):
    """Orthogonalize x in place with an explicit restart schedule: restart
    after each step t in `restarts` (1 <= t < steps); see restart_schedule."""
    _require(x, torch.float32, name="x")
    G, R, C = (1, *x.shape) if x.dim() == 2 else tuple(x.shape)
    keep, cptr = _coeff_array(coeffs, steps)
    mask = 0
    for t in restarts:
        mask |= 1 << int(t)
    lib = load()
    check(lib.gns_orthogonalize_batched_schedule(ctypes.c_void_p(x.data_ptr()), G, R, C, steps, mask, cptr,
                                                 _stream(stream, x.device)), "gns_orthogonalize_batched_schedule")
    del keep
    return x


def gns_gram_ns_state(x, steps=5, restarts=(2,), stream=None):
    """Orthogonalize the rectangular bucket x in place (restart after each
    step in `restarts`) and return the iteration's final Gram state:
    (r_state, q_state, r_scale), two fp16 [G, n, n] device tensors (lower
    triangles defined) with stored R = r_scale * R, and Q unscaled."""
    _require(x, torch.float32, name="x")
    G, R, C = (1, *x.shape) if x.dim() == 2 else tuple(x.shape)
    n = min(R, C)
    r_state = torch.empty(G, n, n, dtype=torch.float16, device=x.device)
    q_state = torch.empty(G, n, n, dtype=torch.float16, device=x.device)
    scale = ctypes.c_float(0.0)
    mask = 0
    for t in restarts:
        mask |= 1 << int(t)
    lib = load()
    check(lib.gns_gram_ns_state(ctypes.c_void_p(x.data_ptr()), G, R, C, steps, mask,
                                ctypes.c_void_p(r_state.data_ptr()), ctypes.c_void_p(q_state.data_ptr()),
                                ctypes.byref(scale), _stream(stream, x.device)), "gns_gram_ns_state")
    return r_state, q_state, float(scale.value)


def gns_orthogonalize_batched_host(x, steps=5, restart_at=2, coeffs=None, stream=None):
    """The same on a host fp32 tensor (pinned memory copies fastest); synchronous."""
    _require(x, torch.float32, cuda=False, name="x")
    G, R, C = (1, *x.shape) if x.dim() == 2 else tuple(x.shape)
    keep, cptr = _coeff_array(coeffs, steps)
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device())
    check(lib.gns_orthogonalize_batched_host(ctypes.c_void_p(x.data_ptr()), G, R, C, steps, restart_at,
                                             cptr, _stream(stream, dev)), "gns_orthogonalize_batched_host")
    del keep
    return x


def gns_orthogonalize_batched_noalloc(x, steps=5, restart_at=2, coeffs=None, stream=None):
    """gns_orthogonalize_batched through the allocation-free entry point: the
    library's workspace is its fixed device array, never cudaMalloc."""
    _require(x, torch.float32, name="x")
    G, R, C = (1, *x.shape) if x.dim() == 2 else tuple(x.shape)
    keep, cptr = _coeff_array(coeffs, steps)
    lib = load()
    check(lib.gns_orthogonalize_batched_noalloc(ctypes.c_void_p(x.data_ptr()), G, R, C, steps, restart_at,
                                                cptr, _stream(stream, x.device)),
          "gns_orthogonalize_batched_noalloc")
    del keep
    return x


def _tensors(ts, dtype, name, base_indices=None):
    arr = (GnsTensor * len(ts))()
    for i, t in enumerate(ts):
        _require(t, dtype, name=name)
        if t.dim() != 2:
            raise ValueError(f"{name}[{i}] must be 2D")
        arr[i].data = t.data_ptr()
        arr[i].rows, arr[i].cols = t.shape
        arr[i].base_index = 0 if base_indices is None else int(base_indices[i])
    return arr


def muon_step(params, grads, momenta, lr, wd, mu, seed, step, base_indices=None, stream=None):
    """One Muon step over lists of bf16 params (in place), bf16 grads and fp32
    momenta (in place). base_indices defaults to the running element offset of
    each parameter, so no two parameters share stochastic-rounding draws."""
    n = len(params)
    if len(grads) != n or len(momenta) != n:
        raise ValueError("params, grads and momenta must have equal lengths")
    if n == 0:
        return
    if base_indices is None:
        base_indices, acc = [], 0
        for p in params:
            base_indices.append(acc)
            acc += p.numel()
    P = _tensors(params, torch.bfloat16, "params", base_indices)
    Gr = _tensors(grads, torch.bfloat16, "grads")
    M = _tensors(momenta, torch.float32, "momenta")
    lib = load()
    check(lib.muon_step(P, Gr, M, n, lr, wd, mu, seed, step, _stream(stream, params[0].device)), "muon_step")


def dion3_step(params, grads, momenta, fraction, lr, wd, mu, seed=0, step=0, base_indices=None, stream=None):
    """One Dion3 step (Algorithm 4, Muon flavor) over lists of bf16 params (in
    place), bf16 grads and fp32 momenta (in place)."""
    n = len(params)
    if len(grads) != n or len(momenta) != n:
        raise ValueError("params, grads and momenta must have equal lengths")
    if n == 0:
        return
    if base_indices is None:
        base_indices, acc = [], 0
        for p in params:
            base_indices.append(acc)
            acc += p.numel()
    P = _tensors(params, torch.bfloat16, "params", base_indices)
    Gr = _tensors(grads, torch.bfloat16, "grads")
    M = _tensors(momenta, torch.float32, "momenta")
    lib = load()
    check(lib.dion3_step(P, Gr, M, n, fraction, lr, wd, mu, seed, step, _stream(stream, params[0].device)),
          "dion3_step")


def normuon_step(params, grads, momenta, second_moments, lr, wd, mu, beta2=0.95, eps=1e-8, seed=0, step=0,
                 base_indices=None, stream=None):
    """One NorMuon step (Dion3 Eq. 2): as muon_step, plus the per-row fp32
    second moments (one float per row of each param, updated in place)."""
    n = len(params)
    if len(grads) != n or len(momenta) != n or len(second_moments) != n:
        raise ValueError("params, grads, momenta and second_moments must have equal lengths")
    if n == 0:
        return
    if base_indices is None:
        base_indices, acc = [], 0
        for p in params:
            base_indices.append(acc)
            acc += p.numel()
    P = _tensors(params, torch.bfloat16, "params", base_indices)
    Gr = _tensors(grads, torch.bfloat16, "grads")
    M = _tensors(momenta, torch.float32, "momenta")
    V = _tensors([v.view(-1, 1) for v in second_moments], torch.float32, "second_moments")
    lib = load()
    check(lib.normuon_step(P, Gr, M, V, n, lr, wd, mu, beta2, eps, seed, step, _stream(stream, params[0].device)),
          "normuon_step")


def gns_muon_momentum(M, G, mu, stream=None):
    """M <- mu M + G (fp32 M in place, bf16 G)."""
    _require(M, torch.float32, name="M")
    _require(G, torch.bfloat16, name="G")
    if M.numel() != G.numel():
        raise ValueError("M and G differ in size")
    lib = load()
    check(lib.gns_muon_momentum(ctypes.c_void_p(M.data_ptr()), ctypes.c_void_p(G.data_ptr()), M.numel(),
                                mu, _stream(stream, M.device)), "gns_muon_momentum")


def gns_muon_update(W, O, lr, wd, scale, seed, step, base_index=0, stream=None):
    """W <- SR_bf16((1 - lr wd) W - lr scale O): W bf16 [R, C] in place, O fp16 [R, C]."""
    _require(W, torch.bfloat16, name="W")
    _require(O, torch.float16, name="O")
    if W.shape != O.shape or W.dim() != 2:
        raise ValueError("W and O must be equal-shaped 2D tensors")
    lib = load()
    check(lib.gns_muon_update(ctypes.c_void_p(W.data_ptr()), ctypes.c_void_p(O.data_ptr()), W.shape[0],
                              W.shape[1], lr, wd, scale, seed, step, base_index, _stream(stream, W.device)),
          "gns_muon_update")


def gns_symm_gemm(A, B, C, D, alpha=1.0, beta=0.0, stream=None):
    """D = alpha A B^T + beta C for symmetric results; fp16 [G, n, k] / [G, n, n]."""
    for t, nm in ((A, "A"), (B, "B"), (D, "D")):
        _require(t, torch.float16, name=nm)
    if C is not None:
        _require(C, torch.float16, name="C")
    G, n, k = A.shape
    lib = load()
    check(lib.gns_symm_gemm(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                            ctypes.c_void_p(C.data_ptr() if C is not None else 0),
                            ctypes.c_void_p(D.data_ptr()), G, n, k, alpha, beta, _stream(stream, A.device)),
          "gns_symm_gemm")
    return D


def gns_get_status(stream=None):
    """Synchronize and return (and clear) the device status word."""
    dev = torch.device("cuda", torch.cuda.current_device())
    return load().gns_get_status(_stream(stream, dev))


def gns_status_string(status):
    return load().gns_status_string(status).decode()


def gns_last_error():
    return load().gns_last_error().decode(errors="replace")


KERNEL_CLASSES = ("gemm_tc", "norm_cast", "muon_elementwise", "copy_rows")


def gns_launch_count():
    """Kernel launches issued by the library since it was loaded."""
    return load().gns_launch_count()


def gns_profile_enable(on=True):
    load().gns_profile_enable(1 if on else 0)


def gns_profile_read():
    """{class: (launches, total ms)} of the profiled launches since the last read."""
    n = len(KERNEL_CLASSES)
    counts = (ctypes.c_int64 * n)()
    ms = (ctypes.c_double * n)()
    check(min(0, load().gns_profile_read(counts, ms, n)), "gns_profile_read")
    return {k: (counts[i], ms[i]) for i, k in enumerate(KERNEL_CLASSES)}


def gns_workspace_bytes():
    return load().gns_workspace_bytes()


def gns_release():
    load().gns_release()

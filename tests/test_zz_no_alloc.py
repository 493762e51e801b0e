"""The allocation-free entry point (for callers whose device memory is held by
their own allocator or pool, or who cannot accept the synchronization of a
workspace allocation) against the allocating gns_orthogonalize_batched.

Collected last on purpose: it runs alone in a fresh process as well as after
every other test."""
import ctypes

import numpy as np
import pytest

from gpu_helpers import assert_parity
from inputs import generators as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from newton_schulz_gram_gb300 import _lib, build
    build.build()
    return _lib.load()


def call_noalloc(lib, t, steps=5, restart_at=2):
    G, R, C = t.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gns_orthogonalize_batched_noalloc(ctypes.c_void_p(t.data_ptr()), G, R, C, steps, restart_at,
                                                 None, stream)


def call_alloc(lib, t, steps=5, restart_at=2):
    G, R, C = t.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gns_orthogonalize_batched(ctypes.c_void_p(t.data_ptr()), G, R, C, steps, restart_at, None, stream)


def test_noalloc_matches_allocating_entry_point_twice_in_a_row(lib):
    cases = [gen.gaussian_bucket(3, 256, 1024, seed=501),   # several matrices per chunk
             gen.gaussian_bucket(2, 1024, 257, seed=502)]   # transposed, ragged, unaligned output rows
    refs = []
    for X in cases:
        t = torch.from_numpy(X).cuda()
        assert call_alloc(lib, t) == 0
        refs.append(t.cpu().numpy())
    torch.cuda.synchronize()

    # Warm-up call: the first call on a device looks up the fixed array.
    w = torch.from_numpy(cases[0]).cuda()
    assert call_noalloc(lib, w) == 0, lib.gns_last_error()
    torch.cuda.synchronize()

    ins = [torch.from_numpy(X).cuda() for X in cases]
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    ws0 = lib.gns_workspace_bytes()
    # Two calls in a row on the same stream, no synchronization between them.
    for t in ins:
        assert call_noalloc(lib, t) == 0, lib.gns_last_error()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert lib.gns_workspace_bytes() == ws0

    for t, ref in zip(ins, refs):
        got = t.cpu().numpy()
        for g in range(got.shape[0]):
            assert_parity(got[g], ref[g], what="noalloc vs gns_orthogonalize_batched")
        assert np.array_equal(got, ref)


def test_noalloc_rejects_too_large_matrices(lib):
    t = torch.empty(1, 4096, 14336, device="cuda")
    assert call_noalloc(lib, t) == -1
    assert "allocation-free" in lib.gns_last_error().decode()

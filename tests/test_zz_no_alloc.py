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


@pytest.mark.parametrize("G,R,C", [(5, 1024, 4096),    # about 26 MB of workspace each: chunks of 2, 2 and 1
                                   (3, 1021, 4093)])   # unaligned rows: staged fp32 output, chunks of 1
def test_noalloc_runs_buckets_larger_than_its_array_in_chunks(lib, G, R, C):
    """A bucket whose workspace exceeds the fixed array runs as several
    sequential chunks that reuse the array; the result equals the allocating
    entry point's bit for bit, with the output written directly into the
    caller's buffer (16-byte rows) and through the staging buffer (other
    rows)."""
    X = gen.gaussian_bucket(G, R, C, seed=503 + C)
    a = torch.from_numpy(X).cuda()
    assert call_alloc(lib, a) == 0
    b = torch.from_numpy(X).cuda()
    assert call_noalloc(lib, b) == 0, lib.gns_last_error()
    torch.cuda.synchronize()
    assert np.array_equal(a.cpu().numpy(), b.cpu().numpy())


def test_noalloc_status_word_is_readable(lib):
    """A non-finite input through the allocation-free entry point is reported
    by gns_get_status (which allocates nothing), and the finite matrices of
    the same bucket are unaffected."""
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.gns_get_status(stream) == 0
    X = gen.gaussian_bucket(3, 256, 1024, seed=504)
    ref = torch.from_numpy(X).cuda()
    assert call_alloc(lib, ref) == 0
    X[1, 0, 0] = np.nan
    t = torch.from_numpy(X).cuda()
    assert call_noalloc(lib, t) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    assert lib.gns_get_status(stream) == -3
    assert lib.gns_get_status(stream) == 0
    assert torch.cuda.mem_get_info()[0] == free0
    got, want = t.cpu().numpy(), ref.cpu().numpy()
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[2], want[2])

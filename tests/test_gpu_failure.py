"""Failure handling on the GPU without a fault: bounded waits that run out, and
a non-finite input matrix inside a bucket of finite ones.

Every device-side wait of the library is bounded. Here a wait is made to run
out on purpose through the library's own check (gns_test_bounded_wait: a
flag that nothing sets, a short bound), never by breaking a kernel: the
kernel returns, the status word says GNS_ERR_TIMEOUT and the next ordinary
call matches the oracle. The pages' only failure mode is numerical
divergence (Dion3 App. B.1), pinned on the CPU by the oracle tests."""
import time

import numpy as np
import pytest

from gpu_helpers import assert_parity
from inputs import generators as gen
from oracle import gram_ns as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GNS_ERR_NONFINITE = -3
GNS_ERR_TIMEOUT = -4


@pytest.fixture(scope="module")
def gns():
    import newton_schulz_gram_gb300 as m
    from newton_schulz_gram_gb300 import build
    build.build()
    m.load()
    return m


def check_against_oracle(gns, X, skip=()):
    t = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32)).cuda()
    gns.gns_orthogonalize_batched(t)
    torch.cuda.synchronize()
    out = t.cpu().numpy()
    for g in range(X.shape[0]):
        if g in skip:
            continue
        assert_parity(out[g], O.orthogonalize(X[g].astype(np.float64)), what=f"matrix {g}")
    return out


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "counter"])
def test_bounded_wait_runs_out_and_the_device_stays_usable(gns, kind):
    import ctypes
    lib = gns.load()
    assert gns.gns_get_status() == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    gave_up = lib.gns_test_bounded_wait(kind, 1_000_000, stream)  # 1 ms for thread 0
    elapsed = time.perf_counter() - t0
    # All 256 waits ended; the 255 with a 1 s bound ended through the abort
    # mark, long before their own bound.
    assert gave_up == 256, gns.gns_last_error()
    assert elapsed < 0.5, elapsed
    assert gns.gns_get_status() == GNS_ERR_TIMEOUT
    assert gns.gns_get_status() == 0
    # The abort mark belongs to the check's call only: an ordinary call after
    # it runs normally.
    check_against_oracle(gns, gen.gaussian_bucket(3, 256, 1024, seed=77))
    assert gns.gns_get_status() == 0


def test_bounded_wait_rejects_bad_arguments(gns):
    import ctypes
    lib = gns.load()
    assert lib.gns_test_bounded_wait(2, 1_000_000, ctypes.c_void_p(0)) == -1
    assert lib.gns_test_bounded_wait(0, 10, ctypes.c_void_p(0)) == -1


def test_nonfinite_matrix_leaves_the_others_intact(gns):
    """One matrix with an infinite entry in a bucket of finite ones: the status
    word records GNS_ERR_NONFINITE, and the finite matrices still match the
    oracle, in this call and in a second one made without reading the status
    word in between (a recorded condition does not make later waits give up)."""
    X = gen.gaussian_bucket(6, 1024, 4096, seed=78)
    X[2, 5, 17] = np.inf
    out = check_against_oracle(gns, X, skip=(2,))
    assert not np.all(np.isfinite(out[2]))
    Y = gen.gaussian_bucket(6, 1024, 4096, seed=79)
    check_against_oracle(gns, Y)
    assert gns.gns_get_status() == GNS_ERR_NONFINITE
    assert gns.gns_get_status() == 0

"""CPU-side checks of the C ABI library: it builds, loads without a GPU,
exports every symbol include/gns.h declares, and rejects bad arguments in
host code (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gns.h")


@pytest.fixture(scope="module")
def lib():
    from newton_schulz_gram_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for must in ("gns_orthogonalize_batched", "muon_step", "gns_symm_gemm", "gns_get_status",
                 "gns_status_string", "gns_release"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from newton_schulz_gram_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.PROTOTYPES, f"binding has no prototype for {name}"


def test_status_strings(lib):
    for code in range(-6, 1):
        assert lib.gns_status_string(code).decode() != "unknown status"
    assert lib.gns_status_string(7).decode() == "unknown status"


def test_bad_arguments_are_rejected_on_the_host(lib):
    vp = ctypes.c_void_p
    assert lib.gns_orthogonalize_batched(vp(0), -1, 4, 4, 5, 2, vp(0), vp(0)) == -1
    assert lib.gns_orthogonalize_batched(vp(0), 1, 0, 4, 5, 2, vp(0), vp(0)) == -1
    assert lib.gns_orthogonalize_batched(vp(0), 1, 4, 4, 0, 2, vp(0), vp(0)) == -1
    assert lib.gns_orthogonalize_batched(vp(0), 1, 4, 4, 65, 2, vp(0), vp(0)) == -1
    assert lib.gns_orthogonalize_batched(vp(0), 1, 4, 4, 5, 2, vp(0), vp(0)) == -1  # null ptr
    assert lib.gns_orthogonalize_batched(vp(0), 0, 4, 4, 5, 2, vp(0), vp(0)) == 0  # empty bucket
    assert lib.gns_symm_gemm(vp(1), vp(1), vp(0), vp(1), 1, 12, 8, 1.0, 0.0, vp(0)) == -1  # n % 8
    assert lib.gns_muon_update(vp(0), vp(0), 4, 4, 0.1, 0.0, 1.0, 0, 0, -1, vp(0)) == -1
    assert lib.muon_step(None, None, None, -1, 0.1, 0.0, 0.9, 0, 0, vp(0)) == -1
    assert lib.muon_step(None, None, None, 0, 0.1, 0.0, 0.9, 0, 0, vp(0)) == 0
    scale = ctypes.c_float(0.0)
    # Gram-state entry: square matrices have no Gram state; mask bits only in 1 .. steps - 1.
    assert lib.gns_gram_ns_state(vp(16), 1, 8, 8, 5, 4, vp(16), vp(16), ctypes.byref(scale), vp(0)) == -1
    assert lib.gns_gram_ns_state(vp(16), 1, 8, 16, 5, 1 << 5, vp(16), vp(16), ctypes.byref(scale), vp(0)) == -1
    assert lib.gns_gram_ns_state(vp(16), 1, 8, 16, 5, 1, vp(16), vp(16), ctypes.byref(scale), vp(0)) == -1
    assert lib.gns_gram_ns_state(vp(16), 1, 8, 16, 5, 4, vp(0), vp(16), ctypes.byref(scale), vp(0)) == -1
    assert lib.gns_last_error().decode() != ""


def test_no_gpu_means_a_loud_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    vp = ctypes.c_void_p
    st = lib.gns_orthogonalize_batched(vp(16), 1, 8, 8, 5, 2, vp(0), vp(0))
    assert st in (-2, -6)

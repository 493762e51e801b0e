"""ctypes loader and prototypes of libgns.so (the C ABI in include/gns.h)."""
from __future__ import annotations

import ctypes
import os
import platform

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", platform.machine(), "libgns.so")

GNS_STATUS = {
    0: "GNS_OK", -1: "GNS_ERR_INVALID", -2: "GNS_ERR_CUDA", -3: "GNS_ERR_NONFINITE",
    -4: "GNS_ERR_TIMEOUT", -5: "GNS_ERR_NOMEM", -6: "GNS_ERR_UNSUPPORTED",
}

# Every symbol include/gns.h declares, with (restype, argtypes).
_vp, _i, _f, _u64, _i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_int64


class GnsTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("rows", ctypes.c_int), ("cols", ctypes.c_int),
                ("base_index", ctypes.c_int64)]


PROTOTYPES = {
    "gns_orthogonalize_batched": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "gns_orthogonalize_batched_schedule": (_i, [_vp, _i, _i, _i, _i, _u64, _vp, _vp]),
    "gns_orthogonalize_batched_host": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "gns_gram_ns_state": (_i, [_vp, _i, _i, _i, _i, _u64, _vp, _vp, ctypes.POINTER(ctypes.c_float), _vp]),
    "gns_orthogonalize_batched_noalloc": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "muon_step": (_i, [ctypes.POINTER(GnsTensor), ctypes.POINTER(GnsTensor), ctypes.POINTER(GnsTensor),
                       _i, _f, _f, _f, _u64, _u64, _vp]),
    "dion3_step": (_i, [ctypes.POINTER(GnsTensor), ctypes.POINTER(GnsTensor), ctypes.POINTER(GnsTensor),
                        _i, _f, _f, _f, _f, _u64, _u64, _vp]),
    "normuon_step": (_i, [ctypes.POINTER(GnsTensor), ctypes.POINTER(GnsTensor), ctypes.POINTER(GnsTensor),
                          ctypes.POINTER(GnsTensor), _i, _f, _f, _f, _f, _f, _u64, _u64, _vp]),
    "gns_muon_momentum": (_i, [_vp, _vp, _i64, _f, _vp]),
    "gns_muon_update": (_i, [_vp, _vp, _i, _i, _f, _f, _f, _u64, _u64, _i64, _vp]),
    "gns_symm_gemm": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _f, _f, _vp]),
    "gns_get_status": (_i, [_vp]),
    "gns_test_bounded_wait": (_i, [_i, _i64, _vp]),
    "gns_status_string": (ctypes.c_char_p, [_i]),
    "gns_last_error": (ctypes.c_char_p, []),
    "gns_workspace_bytes": (_i64, []),
    "gns_launch_count": (_i64, []),
    "gns_profile_enable": (None, [_i]),
    "gns_profile_read": (_i, [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double), _i]),
    "gns_release": (None, []),
}

_LIB = None


class GnsError(RuntimeError):
    def __init__(self, status, where, detail=""):
        self.status = status
        name = GNS_STATUS.get(status, str(status))
        super().__init__(f"{where} failed with {name}" + (f": {detail}" if detail else ""))


def load(path=LIB_PATH):
    """Load libgns.so. Raises if it has not been built: there is no fallback."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libgns.so not found at {path}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'` "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def check(status, where):
    if status != 0:
        lib = load()
        detail = lib.gns_last_error().decode(errors="replace")
        raise GnsError(status, where, detail)
    return status

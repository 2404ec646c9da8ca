"""ctypes binding of libpkd (include/pkd.h).  Argument marshalling only.

The library is loaded from ``paged_kv_decode_23_gb300/_build/libpkd.so`` (built in-tree by
``paged_kv_decode_23_gb300/build.py``).  There is no fallback: if the library is missing or
fails to load, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpkd.so")

PKD_OK = 0
ERRORS = {
    -1: "PKD_ERR_INVALID_ARG",
    -2: "PKD_ERR_NOT_PLANNED",
    -3: "PKD_ERR_WORKSPACE_TOO_SMALL",
    -4: "PKD_ERR_CUDA",
    -5: "PKD_ERR_UNSUPPORTED",
    -6: "PKD_ERR_DEVICE",
}
DTYPE_F16, DTYPE_BF16, DTYPE_E4M3 = 0, 1, 2
LAYOUT_NHD, LAYOUT_HND = 0, 1
KERNEL_AUTO, KERNEL_CUDA_CORE, KERNEL_TENSOR_CORE = -1, 0, 1
STATUS_TIMEOUT, STATUS_BAD_PAGE = 1, 2

# every symbol include/pkd.h declares, with its ctypes signature (pointers, host or device, pass
# as addresses)
_vp = ctypes.c_void_p
_i64p = ctypes.POINTER(ctypes.c_int64)
_c_int, _c_float, _c_size = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "pkd_create": (_c_int, [ctypes.POINTER(_vp), _vp, _c_size, _vp, _c_size, _c_int]),
    "pkd_reset_workspace": (_c_int, [_vp, _vp, _c_size, _vp, _c_size]),
    "pkd_plan": (_c_int, [_vp, _vp, _vp, _c_int, _vp, ctypes.c_int64, _c_int, _c_int, _c_int,
                          _c_int, _c_float, _c_float, _c_int, _c_int, _c_int, _c_int, _c_int,
                          _c_int, _c_int, _c_int, _c_int, _c_float, _c_float, _vp]),
    "pkd_run": (_c_int, [_vp, _vp, _vp, _vp, ctypes.c_int64, _i64p, _c_float, _c_float, _c_float,
                         _vp, _vp, _vp]),
    "pkd_run_timed": (_c_int, [_vp, _vp, _vp, _vp, ctypes.c_int64, _i64p, _c_float, _c_float,
                               _c_float, _vp, _vp, _vp, _vp, _vp]),
    "pkd_destroy": (_c_int, [_vp]),
    "pkd_last_error": (ctypes.c_char_p, []),
    "pkd_workspace_bytes": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                     _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                     ctypes.POINTER(_c_size), ctypes.POINTER(_c_size)]),
    "pkd_plan_host": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                               _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp,
                               _c_int, ctypes.POINTER(_c_int), ctypes.POINTER(_c_int),
                               ctypes.POINTER(_c_int), ctypes.POINTER(_c_int),
                               ctypes.POINTER(_c_int), _c_int, _c_int, ctypes.POINTER(_c_int)]),
    "pkd_check_status": (_c_int, [_vp, ctypes.POINTER(ctypes.c_uint32), _vp]),
    "pkd_set_pdl": (_c_int, [_vp, _c_int]),
    "pkd_set_wait_limit": (_c_int, [_vp, ctypes.c_uint64]),
    "pkd_plan_info": (_c_int, [_vp, ctypes.POINTER(_c_int), ctypes.POINTER(_c_int),
                               ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "pkd_check_page_table": (_c_int, [_vp, _c_int, _vp, ctypes.c_int64, ctypes.c_int64]),
    "pkd_mla_set_backend": (_c_int, [_vp, _c_int]),
    "pkd_mla_plan_host": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                   _vp, _c_int, _vp, _c_int, ctypes.POINTER(_c_int),
                                   ctypes.POINTER(_c_int), ctypes.POINTER(_c_int),
                                   ctypes.POINTER(_c_int), ctypes.POINTER(_c_size),
                                   ctypes.POINTER(_c_size)]),
    "pkd_mla_plan": (_c_int, [_vp, _vp, _vp, _c_int, _vp, ctypes.c_int64, _c_int, _c_int,
                              _c_int, _c_int, _c_int, _c_float, _c_int, _c_int, _vp]),
    "pkd_mla_run": (_c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_int64, _vp, _vp, _c_int, _vp,
                             _vp, _vp]),
    "pkd_enable_cuda_graph": (_c_int, [_vp, _vp, _vp, _vp, _c_int, ctypes.c_int64, _c_int]),
    "pkd_mla_graph_workspace_bytes": (_c_int, [_c_int, _c_int, _c_int, ctypes.POINTER(_c_size),
                                               ctypes.POINTER(_c_size)]),
    "pkd_graph_workspace_bytes": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                           ctypes.POINTER(_c_size), ctypes.POINTER(_c_size)]),
    "pkd_decode_noalloc": (_c_int, [_vp, _vp, _c_int, _vp, ctypes.c_int64, _c_int, _c_int,
                                    _c_int, _c_int, _c_float, _c_float, _c_int, _c_int, _c_int,
                                    _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                    ctypes.c_int64, _i64p, _c_float, _c_float, _c_float, _vp,
                                    _vp, _vp]),
}

_lock = threading.Lock()
_lib = None


class PkdError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def lib():
    """The loaded library; raises if it is not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libpkd is not built ({LIB_PATH} missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(l, name)
                fn.restype = res
                fn.argtypes = args
            _lib = l
    return _lib


def check(rc: int) -> None:
    if rc != PKD_OK:
        raise PkdError(rc, lib().pkd_last_error().decode())

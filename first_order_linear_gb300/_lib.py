"""ctypes view of the C ABI in ``include/rlca.h`` (``librlca.so``).

Only argument marshalling lives here.  :func:`load` opens the in-tree
library built by :mod:`first_order_linear_gb300.build` and raises if it is
missing: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

# RLCA_LIBRARY=checked selects the index-check build of the same sources
# (librlca_checked.so: every call waits for its kernels and fails when one of
# them met an index outside its array); the default is the product build
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                         "librlca_checked.so" if os.environ.get("RLCA_LIBRARY") == "checked" else "librlca.so")
_lock = threading.Lock()
_lib = None

RLCA_OK = 0
RLCA_ERR_INVALID_ARG = 1
RLCA_ERR_UNSUPPORTED = 2
RLCA_ERR_CUDA = 3

RLCA_TIME_MAJOR = 0x1
RLCA_MULTIPASS = 0x2
RLCA_PSUM_EXCLUSIVE = 0x4
RLCA_PSUM_FLAG_IS_START = 0x8
RLCA_INPUTS_READY = 0x10
RLCA_BF16 = 0x20

RLCA_EST_GAE = 1
RLCA_EST_DISCOUNTED_RETURN = 2
RLCA_EST_TD_LAMBDA = 3
RLCA_EST_VTRACE = 4
RLCA_EST_RETRACE = 5
RLCA_EST_ELIG_TRACE = 6
RLCA_EST_PREFIX_SUM = 7
RLCA_EST_AFFINE_SCAN = 8
RLCA_EST_VALUE_TARGETS = 9

RLCA_F32 = 0
RLCA_I32 = 1
RLCA_MAX_ACTIONS = 64
RLCA_STATIC_SCRATCH_BYTES = 1 << 20
RLCA_STATUS_WAIT_TIMEOUT = 0x1
RLCA_STATUS_INDEX = 0x2

_p = C.c_void_p
_i64 = C.c_int64
_u32 = C.c_uint32
_f = C.c_float
_i = C.c_int
_sz = C.c_size_t

# return and argument types of every entry point, in declaration order
SIGNATURES = {
    "rlca_status_string": (C.c_char_p, [_i]),
    "rlca_version": (_i, []),
    "rlca_device_status": (_i, [C.POINTER(C.c_uint), _i]),
    "rlca_index_checks": (_i, []),
    "rlca_workspace_size": (_i, [_i, _i64, _i64, C.c_int32, _u32, C.POINTER(_sz)]),
    "rlca_gae": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _i64, _i64, _f, _f, _u32, _p, _sz, _p]),
    "rlca_value_targets": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i64, _i64, _f, _f, _u32, _p, _sz, _p]),
    "rlca_gae_static_scratch": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _i64, _i64, _f, _f, _u32, _p]),
    "rlca_discounted_return": (_i, [_p, _p, _p, _p, _p, _p, _i64, _i64, _f, _u32, _p, _sz, _p]),
    "rlca_td_lambda": (_i, [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _f, _f, _u32, _p, _sz, _p]),
    "rlca_vtrace": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i64, _i64, _f, _f, _f, _f, _u32, _p, _sz,
                         _p]),
    "rlca_retrace": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i64, _i64, C.c_int32, _f, _f, _u32, _p, _sz,
                          _p]),
    "rlca_elig_trace": (_i, [_p, _p, _p, _p, _i64, _i64, _f, _f, _u32, _p, _sz, _p]),
    "rlca_episodic_prefix_sum": (_i, [_p, _i, _p, _p, _p, _i64, _i64, _u32, _p, _sz, _p]),
    "rlca_affine_scan": (_i, [_p, _p, _p, _p, _i64, _i64, _i, _u32, _p, _sz, _p]),
}


def library_path() -> str:
    return _LIB_PATH


def load() -> C.CDLL:
    """The loaded library with argument types set.  Raises RuntimeError
    when librlca.so has not been built."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with first_order_linear_gb300.build.build() "
                    "(there is no fallback implementation)")
            lib = C.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class RlcaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = load().rlca_status_string(status).decode()
        super().__init__(f"{fn} failed with status {status} ({msg})")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != RLCA_OK:
        raise RlcaError(fn, status)

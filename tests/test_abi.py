"""The C-ABI library without a GPU: it loads, exports every entry point
that include/rlca.h declares, and rejects bad arguments on the host before
touching CUDA (none of these calls reaches the device)."""
import ctypes as C
import os
import re

import pytest

from first_order_linear_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for f in os.listdir(INCLUDE):
        if f.endswith(".h"):
            text = open(os.path.join(INCLUDE, f)).read()
            names.update(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(rlca_\w+)\s*\(", text, re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("rlca_gae", "rlca_vtrace", "rlca_retrace", "rlca_td_lambda", "rlca_discounted_return",
              "rlca_elig_trace", "rlca_episodic_prefix_sum", "rlca_affine_scan", "rlca_workspace_size",
              "rlca_status_string", "rlca_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_host_only_queries(lib):
    assert lib.rlca_version() >= 100
    assert lib.rlca_device_status(None, 0) == _lib.RLCA_ERR_INVALID_ARG
    assert lib.rlca_status_string(0) == b"ok"
    assert lib.rlca_status_string(1) == b"invalid argument"
    assert lib.rlca_status_string(99) == b"unknown status"


FAKE = C.c_void_p(0x10000)       # never dereferenced: every call below fails validation
FAKE2 = C.c_void_p(0x900000)


def gae(lib, **kw):
    a = dict(r=FAKE, v=C.c_void_p(0x200000), term=None, trunc=None, tv=None, boot=None,
             adv=C.c_void_p(0x400000), ret=None, E=4, T=8, flags=0, ws=None, wsb=0)
    a.update(kw)
    return lib.rlca_gae(a["r"], a["v"], a["term"], a["trunc"], a["tv"], a["boot"], a["adv"], a["ret"],
                        a["E"], a["T"], 0.99, 0.95, a["flags"], a["ws"], a["wsb"], None)


def test_empty_call_is_ok(lib):
    assert gae(lib, E=0) == _lib.RLCA_OK
    assert gae(lib, T=0, r=None, v=None, adv=None) == _lib.RLCA_OK


def test_invalid_arguments(lib):
    INV = _lib.RLCA_ERR_INVALID_ARG
    assert gae(lib, E=-1) == INV
    assert gae(lib, T=-5) == INV
    assert gae(lib, T=(1 << 30) + 1) == INV
    assert gae(lib, r=None) == INV
    assert gae(lib, adv=None) == INV
    assert gae(lib, trunc=FAKE2) == INV                      # truncated without trunc_value
    assert gae(lib, flags=0x80) == INV                       # unknown flag
    assert gae(lib, flags=_lib.RLCA_PSUM_EXCLUSIVE) == INV   # prefix-sum flag on GAE
    assert gae(lib, adv=C.c_void_p(0x10000 + 8)) == INV      # output overlaps rewards
    assert gae(lib, ret=C.c_void_p(0x400000 + 64)) == INV    # outputs overlap each other


def test_invalid_arguments_other_entry_points(lib):
    INV, UNS = _lib.RLCA_ERR_INVALID_ARG, _lib.RLCA_ERR_UNSUPPORTED
    P = [C.c_void_p(0x100000 * (i + 1)) for i in range(12)]
    # Retrace: num_actions out of range
    assert lib.rlca_retrace(P[0], P[1], P[2], P[3], P[4], None, None, None, None, P[5], 4, 8, 0,
                            0.99, 0.95, 0, None, 0, None) == INV
    assert lib.rlca_retrace(P[0], P[1], P[2], P[3], P[4], None, None, None, None, P[5], 4, 8, 65,
                            0.99, 0.95, 0, None, 0, None) == UNS
    # prefix sum: unknown dtype
    assert lib.rlca_episodic_prefix_sum(P[0], 7, None, None, P[1], 4, 8, 0, None, 0, None) == INV
    # affine scan: output aliases alpha
    assert lib.rlca_affine_scan(P[0], P[1], None, P[0], 4, 8, 1, 0, None, 0, None) == INV
    # V-Trace: missing log-probs
    assert lib.rlca_vtrace(P[0], P[1], None, P[3], None, None, None, None, P[4], None, 4, 8, 0.99,
                           1.0, 1.0, 1.0, 0, None, 0, None) == INV
    # eligibility trace / discounted return / TD(lambda): missing output
    assert lib.rlca_elig_trace(P[0], None, None, None, 4, 8, 0.99, 0.9, 0, None, 0, None) == INV
    assert lib.rlca_discounted_return(P[0], None, None, None, None, None, 4, 8, 0.99, 0, None, 0, None) == INV
    assert lib.rlca_td_lambda(P[0], P[1], None, None, None, None, None, 4, 8, 0.99, 0.9, 0, None, 0,
                              None) == INV
    # workspace query: bad estimator / NULL output / empty
    out = C.c_size_t(0)
    assert lib.rlca_workspace_size(99, 4, 8, 0, 0, C.byref(out)) == INV
    assert lib.rlca_workspace_size(1, 4, 8, 0, 0, None) == INV
    assert lib.rlca_workspace_size(1, 0, 8, 0, 0, C.byref(out)) == _lib.RLCA_OK and out.value == 0


def test_bf16_flag_scope(lib):
    """RLCA_BF16 covers the float-storage calls; the no-allocation GAE keeps
    float32 (unsupported), int32 prefix sums have no bfloat16 form, and the
    overlap checks count 2-byte elements."""
    INV, UNS, BF = _lib.RLCA_ERR_INVALID_ARG, _lib.RLCA_ERR_UNSUPPORTED, _lib.RLCA_BF16
    P = [C.c_void_p(0x100000 * (i + 1)) for i in range(12)]
    # 4 x 8 x 18 bfloat16 Q values span 1152 bytes: an output 1150 bytes in overlaps them
    assert lib.rlca_retrace(P[0], P[1], P[2], P[3], P[4], None, None, None, None, C.c_void_p(0x100000 + 1150),
                            4, 8, 18, 0.99, 0.95, BF, None, 0, None) == INV
    assert lib.rlca_gae_static_scratch(P[0], P[1], None, None, None, None, P[2], P[3], 4, 8, 0.99, 0.95, BF,
                                       None) == UNS
    assert lib.rlca_episodic_prefix_sum(P[0], _lib.RLCA_I32, None, None, P[1], 4, 8, BF, None, 0, None) == INV
    # 4 x 8 bfloat16 elements span 64 bytes: an output 62 bytes in overlaps the input
    assert lib.rlca_elig_trace(P[0], None, None, C.c_void_p(0x100000 + 62), 4, 8, 0.99, 0.9, BF, None, 0,
                               None) == INV
    out = C.c_size_t(1)
    assert lib.rlca_workspace_size(1, 4, 8, 0, BF, C.byref(out)) in (_lib.RLCA_OK, _lib.RLCA_ERR_CUDA)


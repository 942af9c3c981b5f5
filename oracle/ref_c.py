"""ctypes view of oracle/rlca_ref.c, with the call signatures of
oracle/rlca_ref.py, so the same pins and cross-checks run on both CPU
references.

TEST INFRASTRUCTURE: only the test suite uses this module.  It shares no
code with the CUDA path or with the NumPy reference (it only converts the
inputs to float64 / uint8 / int32 arrays and calls the C loops).
"""
from __future__ import annotations

import ctypes as C
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rlca_ref.c")
LIB = os.path.join(HERE, "librlca_ref.so")

_lib = None


def build() -> str:
    """Compile the C reference (gcc -O2, no fast-math) when it is missing or
    older than its source; returns the library path."""
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found for the C reference")
    tmp = LIB + f".{os.getpid()}.tmp"
    subprocess.run([cc, "-O2", "-std=c99", "-shared", "-fPIC", "-fno-fast-math", SRC, "-o", tmp, "-lm"],
                   check=True)
    os.replace(tmp, LIB)
    return LIB


def load():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        d, u8, i32, i64 = C.POINTER(C.c_double), C.POINTER(C.c_uint8), C.POINTER(C.c_int32), C.c_int64
        sig = {
            "ref_affine_scan": [d, d, d, i64, i64, C.c_int, d],
            "ref_gae": [d, d, u8, u8, d, d, i64, i64, C.c_double, C.c_double, d, d],
            "ref_discounted_return": [d, u8, u8, d, d, i64, i64, C.c_double, d],
            "ref_td_lambda": [d, d, u8, u8, d, d, i64, i64, C.c_double, C.c_double, d],
            "ref_vtrace": [d, d, d, d, u8, u8, d, d, i64, i64, C.c_double, C.c_double, C.c_double, C.c_double,
                           d, d],
            "ref_retrace": [d, d, d, i32, d, u8, u8, d, d, i64, i64, i64, C.c_double, C.c_double, d],
            "ref_eligibility_trace": [d, u8, u8, i64, i64, C.c_double, C.c_double, d],
            "ref_prefix_sum_f64": [d, u8, u8, i64, i64, C.c_int, C.c_int, d],
            "ref_prefix_sum_i32": [i32, u8, u8, i64, i64, C.c_int, C.c_int, i32],
        }
        for name, args in sig.items():
            fn = getattr(_lib, name)
            fn.argtypes = args
            fn.restype = None
    return _lib


# --------------------------------------------------------------------------
# argument conversion (no arithmetic of the method)
# --------------------------------------------------------------------------

def _f(a, shape=None):
    if a is None:
        return None
    x = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None:
        x = x.reshape(shape)
    return x


def _u8(a, shape):
    if a is None:
        return None
    return np.ascontiguousarray((np.asarray(a) != 0).astype(np.uint8).reshape(shape))


def _p(x, ctype):
    return None if x is None else x.ctypes.data_as(C.POINTER(ctype))


def _pd(x):
    return _p(x, C.c_double)


def _check_trunc(truncated, trunc_value):
    if truncated is not None and trunc_value is None:
        raise ValueError("truncated given without trunc_value")


# --------------------------------------------------------------------------
# the estimators, signatures as in oracle/rlca_ref.py
# --------------------------------------------------------------------------

def affine_scan(alpha, beta, carry=None, reverse=True):
    a, b = _f(alpha), _f(beta)
    E, T = a.shape
    out = np.empty((E, T))
    load().ref_affine_scan(_pd(a), _pd(b), _pd(_f(carry, (E,))), E, T, 1 if reverse else 0, _pd(out))
    return out


def gae(rewards, values, terminated, truncated=None, trunc_value=None, bootstrap=None, gamma=0.99, lam=0.95):
    _check_trunc(truncated, trunc_value)
    r, v = _f(rewards), _f(values)
    E, T = r.shape
    adv, ret = np.empty((E, T)), np.empty((E, T))
    load().ref_gae(_pd(r), _pd(v), _p(_u8(terminated, (E, T)), C.c_uint8), _p(_u8(truncated, (E, T)), C.c_uint8),
                   _pd(_f(trunc_value, (E, T))), _pd(_f(bootstrap, (E,))), E, T, gamma, lam, _pd(adv), _pd(ret))
    return adv, ret


def discounted_return(rewards, terminated, truncated=None, trunc_value=None, bootstrap=None, gamma=0.99):
    _check_trunc(truncated, trunc_value)
    r = _f(rewards)
    E, T = r.shape
    out = np.empty((E, T))
    load().ref_discounted_return(_pd(r), _p(_u8(terminated, (E, T)), C.c_uint8),
                                 _p(_u8(truncated, (E, T)), C.c_uint8), _pd(_f(trunc_value, (E, T))),
                                 _pd(_f(bootstrap, (E,))), E, T, gamma, _pd(out))
    return out


def td_lambda(rewards, values, terminated, truncated=None, trunc_value=None, bootstrap=None, gamma=0.99,
              lam=0.95):
    _check_trunc(truncated, trunc_value)
    r, v = _f(rewards), _f(values)
    E, T = r.shape
    out = np.empty((E, T))
    load().ref_td_lambda(_pd(r), _pd(v), _p(_u8(terminated, (E, T)), C.c_uint8),
                         _p(_u8(truncated, (E, T)), C.c_uint8), _pd(_f(trunc_value, (E, T))),
                         _pd(_f(bootstrap, (E,))), E, T, gamma, lam, _pd(out))
    return out


def vtrace(rewards, values, logp_target, logp_behaviour, terminated, truncated=None, trunc_value=None,
           bootstrap=None, gamma=0.99, rho_bar=1.0, c_bar=1.0, lam=1.0):
    _check_trunc(truncated, trunc_value)
    r, v = _f(rewards), _f(values)
    E, T = r.shape
    vs, pg = np.empty((E, T)), np.empty((E, T))
    load().ref_vtrace(_pd(r), _pd(v), _pd(_f(logp_target, (E, T))), _pd(_f(logp_behaviour, (E, T))),
                      _p(_u8(terminated, (E, T)), C.c_uint8), _p(_u8(truncated, (E, T)), C.c_uint8),
                      _pd(_f(trunc_value, (E, T))), _pd(_f(bootstrap, (E,))), E, T, gamma, rho_bar, c_bar, lam,
                      _pd(vs), _pd(pg))
    return vs, pg


def retrace(q, pi, mu_a, actions, rewards, terminated, truncated=None, trunc_value=None, bootstrap=None,
            gamma=0.99, lam=0.95):
    _check_trunc(truncated, trunc_value)
    Q, P = _f(q), _f(pi)
    E, T, A = Q.shape
    r = _f(rewards, (E, T))
    act = np.ascontiguousarray(np.asarray(actions).astype(np.int32).reshape(E, T))
    out = np.empty((E, T))
    load().ref_retrace(_pd(Q), _pd(P), _pd(_f(mu_a, (E, T))), _p(act, C.c_int32), _pd(r),
                       _p(_u8(terminated, (E, T)), C.c_uint8), _p(_u8(truncated, (E, T)), C.c_uint8),
                       _pd(_f(trunc_value, (E, T))), _pd(_f(bootstrap, (E,))), E, T, A, gamma, lam, _pd(out))
    return out


def eligibility_trace(x, terminated, truncated=None, gamma=0.99, lam=0.95):
    xs = _f(x)
    E, T = xs.shape
    out = np.empty((E, T))
    load().ref_eligibility_trace(_pd(xs), _p(_u8(terminated, (E, T)), C.c_uint8),
                                 _p(_u8(truncated, (E, T)), C.c_uint8), E, T, gamma, lam, _pd(out))
    return out


def episodic_prefix_sum(x, terminated, truncated=None, exclusive=False, flag_is_start=False):
    xv = np.asarray(x)
    E, T = xv.shape
    term, trunc = _u8(terminated, (E, T)), _u8(truncated, (E, T))
    if np.issubdtype(xv.dtype, np.integer):
        xi = np.ascontiguousarray((xv.astype(np.int64) & 0xFFFFFFFF).astype(np.uint32).view(np.int32))
        out = np.empty((E, T), dtype=np.int32)
        load().ref_prefix_sum_i32(_p(xi, C.c_int32), _p(term, C.c_uint8), _p(trunc, C.c_uint8), E, T,
                                  int(exclusive), int(flag_is_start), _p(out, C.c_int32))
        return out
    xs = _f(xv)
    out = np.empty((E, T))
    load().ref_prefix_sum_f64(_pd(xs), _p(term, C.c_uint8), _p(trunc, C.c_uint8), E, T, int(exclusive),
                              int(flag_is_start), _pd(out))
    return out

"""rlca_gae_static_scratch: GAE for callers that cannot allocate device memory.

Some callers of this library have no way to allocate the workspace that the
two-pass path needs (a C host linked only against the library, a simulator
callback that must not touch the device heap, a process that reserved all
device memory at start-up).  This entry point uses scratch that the library
itself keeps in device memory instead.  These tests call it through the C
ABI on problems that take the two-pass path, twice in a row with different
inputs (the scratch keeps the previous call's contents), and compare each
result with rlca_gae given an ordinary workspace, at the tolerance of the
other parity tests.  They also check that a problem needing more scratch than
the library holds is refused without touching the outputs.
"""
import ctypes as C

import pytest
import torch

from first_order_linear_gb300 import _lib, rlca
from tests import parity

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _static_call(lib, d, time_major, multipass, adv, ret):
    E, T = (d["rewards"].shape[1], d["rewards"].shape[0]) if time_major else d["rewards"].shape
    flags = (_lib.RLCA_TIME_MAJOR if time_major else 0) | (_lib.RLCA_MULTIPASS if multipass else 0)
    return lib.rlca_gae_static_scratch(
        _p(d["rewards"]), _p(d["values"]), _p(d["terminated"]), _p(d["truncated"]), _p(d["trunc_value"]),
        _p(d["bootstrap"]), _p(adv), _p(ret), E, T, parity.GAMMA, parity.LAMBDA, flags,
        C.c_void_p(torch.cuda.current_stream().cuda_stream))


def _compare(a, b, what):
    err = ((a.double() - b.double()).abs() / (1.0 + b.double().abs())).max().item()
    assert err <= parity.TOL, f"{what}: max rel err {err:.3e}"


CASES = [
    # (E, T, time_major, multipass): each takes the two-pass path
    (5, 40000, False, False),
    (64, 512, False, True),
    (40, 3000, True, False),
    (33, 777, True, True),
]


@pytest.mark.parametrize("E,T,tm,mp", CASES)
def test_static_scratch_matches_workspace_path(cuda_lib, E, T, tm, mp):
    flags = (_lib.RLCA_TIME_MAJOR if tm else 0) | (_lib.RLCA_MULTIPASS if mp else 0)
    need = rlca.rlca_workspace_size(_lib.RLCA_EST_GAE, E, T, flags=flags)
    assert 0 < need <= _lib.RLCA_STATIC_SCRATCH_BYTES, need   # the scratch is really used
    for call, seed in enumerate((101, 202)):
        d = parity.make_inputs("gae", E, T, seed=seed + E + T, trunc=True, device="cuda", p_term=0.02)
        x = parity._tm(d, tm)
        shape = tuple(x["rewards"].shape)
        adv = torch.full(shape, float("nan"), device="cuda")
        ret = torch.full(shape, float("nan"), device="cuda")
        status = _static_call(cuda_lib, x, tm, mp, adv, ret)
        assert status == _lib.RLCA_OK, cuda_lib.rlca_status_string(status)
        ref_adv, ref_ret = rlca.rlca_gae(x["rewards"], x["values"], x["terminated"], x["truncated"],
                                         x["trunc_value"], x["bootstrap"], gamma=parity.GAMMA,
                                         lambda_=parity.LAMBDA, time_major=tm, multipass=mp)
        torch.cuda.synchronize()
        _compare(adv, ref_adv, f"advantages, call {call + 1}")
        _compare(ret, ref_ret, f"returns, call {call + 1}")


@pytest.mark.parametrize("tm", [False, True], ids=["env_major", "time_major"])
def test_static_scratch_single_pass_needs_no_scratch(cuda_lib, tm):
    """4096 x 128 takes the one-pass drivers: the entry point must work
    without ever looking at its scratch."""
    E, T = 4096, 128
    flags = _lib.RLCA_TIME_MAJOR if tm else 0
    assert rlca.rlca_workspace_size(_lib.RLCA_EST_GAE, E, T, flags=flags) == 0
    for call, seed in enumerate((303, 404)):
        d = parity.make_inputs("gae", E, T, seed=seed, trunc=True, device="cuda")
        x = parity._tm(d, tm)
        shape = tuple(x["rewards"].shape)
        adv = torch.full(shape, float("nan"), device="cuda")
        ret = torch.full(shape, float("nan"), device="cuda")
        status = _static_call(cuda_lib, x, tm, False, adv, ret)
        assert status == _lib.RLCA_OK, cuda_lib.rlca_status_string(status)
        ref_adv, ref_ret = rlca.rlca_gae(x["rewards"], x["values"], x["terminated"], x["truncated"],
                                         x["trunc_value"], x["bootstrap"], gamma=parity.GAMMA,
                                         lambda_=parity.LAMBDA, time_major=tm)
        torch.cuda.synchronize()
        _compare(adv, ref_adv, f"advantages, call {call + 1}")
        _compare(ret, ref_ret, f"returns, call {call + 1}")


def test_static_scratch_refuses_oversized_problems(cuda_lib):
    # time-major, forced two pass: 2100 rows x 64 segments x 8 B > 1 MiB
    E, T = 2100, 8192
    flags = _lib.RLCA_TIME_MAJOR | _lib.RLCA_MULTIPASS
    assert rlca.rlca_workspace_size(_lib.RLCA_EST_GAE, E, T, flags=flags) > _lib.RLCA_STATIC_SCRATCH_BYTES
    d = parity.make_inputs("gae", E, T, seed=7, trunc=False, device="cuda")
    x = parity._tm(d, True)
    adv = torch.full((T, E), float("nan"), device="cuda")
    status = _static_call(cuda_lib, x, True, True, adv, None)
    torch.cuda.synchronize()
    assert status == _lib.RLCA_ERR_UNSUPPORTED
    assert torch.isnan(adv).all()

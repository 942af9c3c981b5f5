"""The index-check build (librlca_checked.so, compiled with RLCA_INDEX_CHECK).

Its kernels check every global and shared-memory index of the staged, bulk
(tensor-copy) and two-pass paths -- loads, stores, ring and stage offsets,
segment maps, Retrace's staged scalars and scalar planes -- and record a
miss in a device status word instead of trapping; every call then waits for
its kernels and returns RLCA_ERR_CUDA if any recorded something.  A fresh
process selects that build (RLCA_LIBRARY=checked) and runs ragged,
unaligned, two-pass, time-major and Retrace cases against the oracle: each
call must return RLCA_OK, match the oracle, and leave the status word 0.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import ctypes as C, json, sys
sys.path.insert(0, ROOT)
import torch
from first_order_linear_gb300 import _lib, build
build.build()
lib = _lib.load()
assert lib.rlca_index_checks() == 1, "not the index-check build"
from tests import parity
cases = [
    # (kind, E, T, time_major, multipass, shift): ragged, unaligned, two-pass, tiles and stages
    ("gae", 37, 129, False, False, False), ("vt", 37, 129, True, False, False),
    ("vtrace", 33, 100, False, False, True), ("td", 48, 64, True, False, True),
    ("gae", 64, 512, False, True, False), ("vt", 64, 2048, True, True, False),
    ("disc", 3, 40000, False, False, False), ("elig", 3, 40000, True, False, False),
    ("psum_i32", 256, 2048, True, False, False), ("affine_bwd", 96, 520, True, False, False),
    ("vtrace", 1024, 512, True, False, False), ("gae", 16384, 256, True, False, False),
    ("vt", 4096, 128, False, False, False), ("gae", 4096, 2048, True, False, False),
    ("retrace", 20, 700, False, True, False), ("retrace", 70, 300, True, True, False),
    ("retrace", 3, 40000, True, False, False), ("retrace", 33, 130, False, False, True),
    ("retrace", 1000, 1000, True, False, False), ("retrace", 13, 2048, True, False, True),
    ("gae", 2432, 1032, True, False, False), ("vtrace", 4096, 1024, True, False, False),
    ("vtrace", 9744, 64, True, False, False), ("vt", 10240, 520, True, False, False),
]
worst = 0.0
for kind, E, T, tm, mp, shift in cases:
    worst = max(worst, parity.check_case(kind, E, T, seed=E * 7 + T, time_major=tm, multipass=mp, shift=shift))
st = C.c_uint(0)
assert lib.rlca_device_status(C.byref(st), 0) == 0
print(json.dumps({"cases": len(cases), "worst": worst, "status": st.value}))
"""


def test_index_check_build_runs_clean():
    env = dict(os.environ, RLCA_LIBRARY="checked")
    res = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + SCRIPT], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    out = json.loads(res.stdout.strip().splitlines()[-1])
    assert out["status"] == 0 and out["cases"] >= 20
    assert out["worst"] <= 1e-4

"""The launch planner without a GPU: tests/planner_check.cu, compiled against
the built library, plans a grid of estimators, sizes, layouts, storage types
and pointer alignments and checks what the drivers rely on (rows, tiles and
segments cover the problem, shared memory fits, workspace sizes, the shapes
the fast, staged and tensor-copy drivers assume).  The planner is host code,
so nothing here touches CUDA."""
import os
import re
import shutil
import subprocess

import pytest

from first_order_linear_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    lib = build.build(variants=("product",))
    libdir = os.path.dirname(lib)
    exe = str(tmp_path_factory.mktemp("planner") / "planner_check")
    cmd = [nvcc, "-std=c++17", "-O1", "-diag-suppress", "1886", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(libdir, "csrc"), "-gencode", "arch=compute_103a,code=sm_103a",
           os.path.join(ROOT, "tests", "planner_check.cu"), lib, "-Xlinker", "-rpath," + libdir, "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, timeout=600)
    return exe


def test_planner_invariants(harness):
    out = subprocess.run([harness], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout[-3000:]
    m = re.search(r"planner ok (\d+) fast (\d+) tm_fast (\d+) staged (\d+) bulk (\d+) two_pass (\d+) "
                  r"retrace_tail (\d+)", out.stdout)
    assert m, out.stdout
    total, *per_driver = (int(x) for x in m.groups())
    assert total > 20000
    # the grid reaches every driver the planner can choose
    assert all(n > 0 for n in per_driver), out.stdout

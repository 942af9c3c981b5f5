"""The vectorised PyTorch doubling-scan baseline that ``bench.py
--torch-baseline`` times beside the library computes the same estimators:
checked here on the CPU against the float64 oracle (float32 within the
parity bound, int32 bit-exact), so its timings compare like with like."""
import numpy as np
import pytest

import bench
from tests import parity

KINDS = ["vt", "gae", "disc", "td", "vtrace", "retrace", "elig", "psum"]


@pytest.mark.parametrize("trunc", [False, True], ids=["no_trunc", "trunc"])
@pytest.mark.parametrize("E,T", [(7, 45), (3, 1), (2, 64)])
@pytest.mark.parametrize("kind", KINDS)
def test_torch_doubling_matches_oracle(kind, E, T, trunc):
    pk = "psum_i32" if kind == "psum" else kind
    d = parity.make_inputs(pk, E, T, seed=E * 17 + T, trunc=trunc, device="cpu", p_term=0.05)
    got = bench.torch_doubling(kind, d, gamma=parity.GAMMA, lam=parity.LAMBDA)
    want = parity.run_oracle(pk, d, rows=None)
    assert len(got) == len(want)
    for i, (g, w) in enumerate(zip(got, want)):
        g = g.numpy()
        if kind == "psum":
            assert g.dtype == np.int32 and np.array_equal(g, w), f"psum out{i}"
        else:
            parity.assert_close(g, w, f"{kind} out{i} E={E} T={T} trunc={trunc}", tol=parity.TOL)


def test_doubling_scan_is_the_recurrence():
    """The doubling passes against the serial recurrence on random maps,
    both directions, including T not a power of two."""
    import torch
    g = torch.Generator().manual_seed(5)
    a, b = torch.randn(4, 37, generator=g, dtype=torch.float64), torch.rand(4, 37, generator=g, dtype=torch.float64)
    for reverse in (True, False):
        want = torch.empty_like(a)
        acc = torch.zeros(4, dtype=torch.float64)
        for k in range(37):
            t = 36 - k if reverse else k
            acc = a[:, t] + b[:, t] * acc
            want[:, t] = acc
        assert torch.allclose(bench.torch_doubling_scan(a, b, reverse=reverse), want, rtol=1e-12, atol=1e-12)

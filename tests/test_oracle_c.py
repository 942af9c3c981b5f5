"""The second CPU reference (plain C, oracle/rlca_ref.c) against the same
pins as the NumPy one, and the two references against each other on seeded
rollouts with every boundary case: two implementations written separately
from the definitions, agreeing to float64 rounding."""
import numpy as np
import pytest

from oracle import ref_c, rlca_ref
from tests import pins


@pytest.fixture(scope="module", autouse=True)
def _built():
    ref_c.build()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin_on_c_reference(pin):
    pin(ref_c)


def _rollout(seed, E=9, T=37, A=5, p_term=0.15, p_trunc=0.12):
    rng = np.random.default_rng(seed)
    term = rng.random((E, T)) < p_term
    trunc = rng.random((E, T)) < p_trunc  # overlaps term on purpose: termination must win
    logits_t, logits_b = rng.normal(size=(E, T, A)), rng.normal(size=(E, T, A))
    pi = np.exp(logits_t) / np.exp(logits_t).sum(-1, keepdims=True)
    mu = np.exp(logits_b) / np.exp(logits_b).sum(-1, keepdims=True)
    act = rng.integers(0, A, size=(E, T))
    return dict(r=rng.normal(size=(E, T)), v=rng.normal(size=(E, T)), tv=rng.normal(size=(E, T)),
                b=rng.normal(size=E), term=term, trunc=trunc, lp=rng.normal(size=(E, T)) * 0.5,
                lb=rng.normal(size=(E, T)) * 0.5, q=rng.normal(size=(E, T, A)), pi=pi,
                mu_a=np.take_along_axis(mu, act[..., None], -1)[..., 0], act=act,
                x=rng.normal(size=(E, T)), xi=rng.integers(-2**31, 2**31, size=(E, T)).astype(np.int32))


def _close(a, b):
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_references_agree(seed):
    d = _rollout(seed)
    for with_trunc in (True, False):
        tr, tv = (d["trunc"], d["tv"]) if with_trunc else (None, None)
        for mod_args in [("gae", (d["r"], d["v"], d["term"], tr, tv, d["b"]), dict(gamma=0.97, lam=0.9)),
                         ("discounted_return", (d["r"], d["term"], tr, tv, d["b"]), dict(gamma=0.97)),
                         ("td_lambda", (d["r"], d["v"], d["term"], tr, tv, d["b"]), dict(gamma=0.97, lam=0.9)),
                         ("vtrace", (d["r"], d["v"], d["lp"], d["lb"], d["term"], tr, tv, d["b"]),
                          dict(gamma=0.97, rho_bar=1.0, c_bar=0.9, lam=0.95)),
                         ("retrace", (d["q"], d["pi"], d["mu_a"], d["act"], d["r"], d["term"], tr, tv, d["b"]),
                          dict(gamma=0.97, lam=0.9)),
                         ("eligibility_trace", (d["x"], d["term"], tr), dict(gamma=0.97, lam=0.9))]:
            name, args, kw = mod_args
            got, want = getattr(ref_c, name)(*args, **kw), getattr(rlca_ref, name)(*args, **kw)
            for g, w in zip(got if isinstance(got, tuple) else (got,), want if isinstance(want, tuple) else (want,)):
                _close(g, w)
        for excl in (False, True):
            for start in (False, True):
                _close(ref_c.episodic_prefix_sum(d["x"], d["term"], tr, exclusive=excl, flag_is_start=start),
                       rlca_ref.episodic_prefix_sum(d["x"], d["term"], tr, exclusive=excl, flag_is_start=start))
                gi = ref_c.episodic_prefix_sum(d["xi"], d["term"], tr, exclusive=excl, flag_is_start=start)
                wi = rlca_ref.episodic_prefix_sum(d["xi"], d["term"], tr, exclusive=excl, flag_is_start=start)
                assert gi.dtype == np.int32 and np.array_equal(gi, wi)
    for rev in (True, False):
        _close(ref_c.affine_scan(d["x"], d["v"] * 0.5, d["b"], reverse=rev),
               rlca_ref.affine_scan(d["x"], d["v"] * 0.5, d["b"], reverse=rev))

"""Pins of the float64 oracle to facts outside itself.

Each ``pin_*`` function takes the oracle module and raises AssertionError
when the oracle disagrees with something the rl-triton paper
(arXiv:2608.17641) or the primary definitions it cites fix independently:

* closed forms (constant reward, x = 1 counters, geometric traces),
* special cases that reduce to a textbook estimator (lambda = 0 / 1 limits,
  on-policy V-Trace, lambda = 0 Retrace = expected-SARSA target),
* the explicit-sum ("forward view") definitions written as brute-force
  double loops on tiny inputs (GAE as a sum of discounted TD errors
  [Schulman et al., 2016]; the lambda-return as a weighted sum of n-step
  returns; V-Trace's sum of clipped TD errors [Espeholt et al., 2018];
  Retrace's sum of traced TD errors [Munos et al., 2016]),
* the worked four-thread scan trace of the paper's Appendix A,
* the no-leak invariant of §5 Correctness Analysis (nothing after an
  episode boundary reaches a step before it, and vice versa for the forward
  scans).

The functions are parametrised by the module so that a planted mistake in
a copy of the oracle can be shown to fail at least one of them.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# brute-force helpers, written from the explicit-sum definitions
# --------------------------------------------------------------------------

def _episode_end(term, trunc, t, T):
    """Last step of the stretch that starts at t: the first k >= t with a
    termination or truncation, else the last step of the window."""
    k = t
    while k < T - 1 and not (term[k] or trunc[k]):
        k += 1
    return k


def _edge_value(k, T, term, trunc, tv, b):
    """Value the step k bootstraps from at the end of a stretch (termination
    wins over truncation; the window edge takes the bootstrap)."""
    if term[k]:
        return 0.0
    if trunc[k]:
        return tv[k]
    assert k == T - 1
    return b


def _random_rollout(rng, E, T, p_term=0.15, p_trunc=0.12):
    """Small random rollout; flags drawn independently, so some steps carry
    both (termination must win)."""
    return dict(
        r=rng.normal(size=(E, T)), v=rng.normal(size=(E, T)),
        term=(rng.random((E, T)) < p_term).astype(np.uint8),
        trunc=(rng.random((E, T)) < p_trunc).astype(np.uint8),
        tv=rng.normal(size=(E, T)), b=rng.normal(size=E))


def _close(got, want, tol=1e-11, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.max(np.abs(got - want) / (1.0 + np.abs(want))) if got.size else 0.0
    assert got.shape == want.shape and err <= tol, f"{what}: max rel err {err}"


# --------------------------------------------------------------------------
# the recurrence
# --------------------------------------------------------------------------

def pin_affine_closed_form(ref):
    """A_t as the explicit product-sum of the recurrence (both directions)."""
    rng = np.random.default_rng(11)
    for T in (1, 2, 3, 5, 8):
        E = 3
        al = rng.normal(size=(E, T))
        be = rng.uniform(-1.3, 1.3, size=(E, T))
        be[rng.random((E, T)) < 0.2] = 0.0
        c = rng.normal(size=E)
        back = ref.affine_scan(al, be, c, reverse=True)
        fwd = ref.affine_scan(al, be, c, reverse=False)
        wb = np.zeros((E, T))
        wf = np.zeros((E, T))
        for e in range(E):
            for t in range(T):
                wb[e, t] = sum(np.prod(be[e, t:k]) * al[e, k] for k in range(t, T)) \
                    + np.prod(be[e, t:T]) * c[e]
                wf[e, t] = sum(np.prod(be[e, k + 1:t + 1]) * al[e, k] for k in range(t + 1)) \
                    + np.prod(be[e, 0:t + 1]) * c[e]
        _close(back, wb, what=f"backward T={T}")
        _close(fwd, wf, what=f"forward T={T}")


def _combine(outer, inner):
    """The paper's combine (§Methodology / §2.2): (aB, bB) (+) (aA, bA) =
    (aB + bB*aA, bA*bB), B the tuple whose timestep comes first in the scan
    direction's output order (the outer map)."""
    aB, bB = outer
    aA, bA = inner
    return (aB + bB * aA, bA * bB)


def pin_combine_algebra(ref):
    """The combine of §2.2 is associative ((X+Y)+Z = X+(Y+Z) on random
    tuples), has the identity (0, 1), and a reset (alpha, 0) absorbs what it
    is composed with (§5: beta = 0 severs the carry); and the oracle's
    recurrence over a row equals the combine of its recurrences over the two
    parts of any split of the row (the regrouping every parallel scan relies
    on).  A segment's map is (A with carry 0, change of A per unit carry)."""
    rng = np.random.default_rng(21)
    for _ in range(200):
        X, Y, Z = (tuple(rng.normal(size=2)) for _ in range(3))
        _close(np.array(_combine(_combine(X, Y), Z)), np.array(_combine(X, _combine(Y, Z))), tol=1e-12,
               what="associativity")
        _close(np.array(_combine(X, (0.0, 1.0))), np.array(X), tol=1e-15, what="right identity")
        _close(np.array(_combine((0.0, 1.0), X)), np.array(X), tol=1e-15, what="left identity")
        _close(np.array(_combine((X[0], 0.0), Y)), np.array((X[0], 0.0)), tol=1e-15, what="reset absorbs")
    for T in (2, 5, 9):
        a = rng.normal(size=(1, T))
        b = rng.uniform(-1.2, 1.2, size=(1, T))

        def seg_map(lo, hi):
            zero = ref.affine_scan(a[:, lo:hi], b[:, lo:hi], np.zeros(1), reverse=True)[0, 0]
            one = ref.affine_scan(a[:, lo:hi], b[:, lo:hi], np.ones(1), reverse=True)[0, 0]
            return (zero, one - zero)

        whole = seg_map(0, T)
        for k in range(1, T):
            _close(np.array(_combine(seg_map(0, k), seg_map(k, T))), np.array(whole), tol=1e-10,
                   what=f"split T={T} at {k}")


def load_app_a_trace():
    rows = []
    with open(os.path.join(GOLDEN, "app_a_four_thread_trace.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            label, span, alpha, beta = [p.strip() for p in line.split("|")]
            lo, hi = (int(x) for x in span.split())
            rows.append((label, lo, hi, alpha, beta))
    return rows


def pin_app_a_trace(ref):
    """The four-thread trace of Appendix A: each printed tuple equals the
    oracle's recurrence over the timesteps it spans (alpha part = result
    with zero carry, beta part = change per unit of carry), and thread 4's
    tuple after the stride-2 pass covers all four timesteps."""
    rng = np.random.default_rng(12)
    rows = load_app_a_trace()
    for trial in range(5):
        a = rng.normal(size=4)
        b = rng.uniform(-1.5, 1.5, size=4)
        env = {f"a{k}": a[k] for k in range(4)}
        env.update({f"b{k}": b[k] for k in range(4)})
        tuples = {}
        for label, lo, hi, ae, bexpr in rows:
            if ae.startswith("COMBINE"):
                x, y = ae[len("COMBINE("):-1].split(",")
                al, be = _combine(tuples[x.strip()], tuples[y.strip()])
            else:
                al = eval(ae, {"__builtins__": {}}, env)
                be = eval(bexpr, {"__builtins__": {}}, env)
            tuples[label] = (al, be)
            seg_a = a[lo:hi + 1][None, :]
            seg_b = b[lo:hi + 1][None, :]
            zero = ref.affine_scan(seg_a, seg_b, np.zeros(1), reverse=True)[0, 0]
            one = ref.affine_scan(seg_a, seg_b, np.ones(1), reverse=True)[0, 0]
            _close(zero, al, what=f"{label} alpha")
            _close(one - zero, be, tol=1e-10, what=f"{label} beta")


# --------------------------------------------------------------------------
# discounted return
# --------------------------------------------------------------------------

def pin_discounted_closed_form(ref):
    """Constant reward c, no boundaries: G_t = c (1 - g^(T-t)) / (1 - g)
    + g^(T-t) * bootstrap."""
    E, T, c, g = 3, 37, 0.7, 0.97
    b = np.array([0.0, 1.5, -2.0])
    r = np.full((E, T), c)
    got = ref.discounted_return(r, np.zeros((E, T), np.uint8), bootstrap=b, gamma=g)
    t = np.arange(T)
    want = c * (1 - g ** (T - t))[None, :] / (1 - g) + (g ** (T - t))[None, :] * b[:, None]
    _close(got, want, what="discounted closed form")


def pin_discounted_bruteforce(ref):
    rng = np.random.default_rng(13)
    g = 0.9
    for T in (1, 2, 4, 6):
        d = _random_rollout(rng, 6, T)
        got = ref.discounted_return(d["r"], d["term"], d["trunc"], d["tv"], d["b"], gamma=g)
        want = np.zeros_like(got)
        for e in range(6):
            term, trunc = d["term"][e], d["trunc"][e]
            for t in range(T):
                k = _episode_end(term, trunc, t, T)
                want[e, t] = sum(g ** (j - t) * d["r"][e, j] for j in range(t, k + 1)) \
                    + g ** (k - t + 1) * _edge_value(k, T, term, trunc, d["tv"][e], d["b"][e])
        _close(got, want, what=f"discounted brute force T={T}")


# --------------------------------------------------------------------------
# GAE
# --------------------------------------------------------------------------

def _td_errors(d, e, T, g):
    """One-step TD errors delta_k of row e: r_k + g * next - v_k, with next
    = v_{k+1} inside a stretch and the edge value at its end."""
    term, trunc = d["term"][e], d["trunc"][e]
    out = np.zeros(T)
    for k in range(T):
        end = _episode_end(term, trunc, k, T)
        nxt = d["v"][e, k + 1] if k < end else _edge_value(k, T, term, trunc, d["tv"][e], d["b"][e])
        out[k] = d["r"][e, k] + g * nxt - d["v"][e, k]
    return out


def pin_gae_bruteforce(ref):
    """A_t = sum_l (g*lam)^l delta_{t+l} over the rest of t's stretch."""
    rng = np.random.default_rng(14)
    g, lam = 0.93, 0.8
    for T in (1, 2, 3, 6):
        d = _random_rollout(rng, 6, T)
        adv, ret = ref.gae(d["r"], d["v"], d["term"], d["trunc"], d["tv"], d["b"], gamma=g, lam=lam)
        want = np.zeros_like(adv)
        for e in range(6):
            delta = _td_errors(d, e, T, g)
            for t in range(T):
                k = _episode_end(d["term"][e], d["trunc"][e], t, T)
                want[e, t] = sum((g * lam) ** (j - t) * delta[j] for j in range(t, k + 1))
        _close(adv, want, what=f"GAE brute force T={T}")
        _close(ret, want + d["v"], what=f"GAE returns T={T}")


def pin_gae_lambda_limits(ref):
    """lam = 0: the advantage is the one-step TD error; lam = 1: it is the
    discounted return minus the value."""
    rng = np.random.default_rng(15)
    g = 0.95
    E, T = 5, 9
    d = _random_rollout(rng, E, T)
    adv0, _ = ref.gae(d["r"], d["v"], d["term"], d["trunc"], d["tv"], d["b"], gamma=g, lam=0.0)
    want0 = np.stack([_td_errors(d, e, T, g) for e in range(E)])
    _close(adv0, want0, what="GAE lam=0")
    adv1, _ = ref.gae(d["r"], d["v"], d["term"], d["trunc"], d["tv"], d["b"], gamma=g, lam=1.0)
    G = ref.discounted_return(d["r"], d["term"], d["trunc"], d["tv"], d["b"], gamma=g)
    _close(adv1, G - d["v"], what="GAE lam=1")


# --------------------------------------------------------------------------
# TD(lambda)
# --------------------------------------------------------------------------

def pin_td_lambda_forward_view(ref):
    """lambda-return as the weighted mix of n-step returns:
    G^lam_t = (1-lam) sum_{n=1}^{N-1} lam^(n-1) G^(n)_t + lam^(N-1) G^(N)_t,
    N = steps to the end of t's stretch, G^(n) bootstrapped from V_{t+n}
    (from the edge value for n = N)."""
    rng = np.random.default_rng(16)
    g, lam = 0.9, 0.7
    for T in (1, 2, 4, 6):
        d = _random_rollout(rng, 5, T)
        got = ref.td_lambda(d["r"], d["v"], d["term"], d["trunc"], d["tv"], d["b"], gamma=g, lam=lam)
        want = np.zeros_like(got)
        for e in range(5):
            term, trunc = d["term"][e], d["trunc"][e]
            for t in range(T):
                k = _episode_end(term, trunc, t, T)
                N = k - t + 1
                edge = _edge_value(k, T, term, trunc, d["tv"][e], d["b"][e])

                def nstep(n):
                    boot = d["v"][e, t + n] if n < N else edge
                    return sum(g ** i * d["r"][e, t + i] for i in range(n)) + g ** n * boot

                want[e, t] = (1 - lam) * sum(lam ** (n - 1) * nstep(n) for n in range(1, N)) \
                    + lam ** (N - 1) * nstep(N)
        _close(got, want, what=f"TD(lambda) forward view T={T}")


def pin_td_lambda_is_gae_return(ref):
    rng = np.random.default_rng(17)
    d = _random_rollout(rng, 7, 11)
    td = ref.td_lambda(d["r"], d["v"], d["term"], d["trunc"], d["tv"], d["b"], gamma=0.97, lam=0.6)
    _, ret = ref.gae(d["r"], d["v"], d["term"], d["trunc"], d["tv"], d["b"], gamma=0.97, lam=0.6)
    _close(td, ret, what="TD(lambda) == GAE return")


# --------------------------------------------------------------------------
# V-Trace
# --------------------------------------------------------------------------

def _vtrace_inputs(rng, E, T):
    d = _random_rollout(rng, E, T)
    d["lp"] = rng.normal(scale=0.8, size=(E, T))
    d["lm"] = rng.normal(scale=0.8, size=(E, T))
    return d


def pin_vtrace_bruteforce(ref):
    """vs_s = V_s + sum_{t=s}^{end} g^(t-s) (prod_{i=s}^{t-1} c_i) delta_t,
    delta_t = rho_t (r_t + g * next_t - V_t); pg_s = rho_s (r_s + g * vs_next
    - V_s).  rho_bar != c_bar and lam != 1 so that the clips are told
    apart."""
    rng = np.random.default_rng(18)
    g, rho_bar, c_bar, lam = 0.92, 1.3, 0.7, 0.9
    for T in (1, 2, 3, 6):
        d = _vtrace_inputs(rng, 6, T)
        vs, pg = ref.vtrace(d["r"], d["v"], d["lp"], d["lm"], d["term"], d["trunc"], d["tv"], d["b"],
                            gamma=g, rho_bar=rho_bar, c_bar=c_bar, lam=lam)
        wvs = np.zeros_like(vs)
        wpg = np.zeros_like(pg)
        for e in range(6):
            term, trunc = d["term"][e], d["trunc"][e]
            ratio = [np.exp(d["lp"][e, t] - d["lm"][e, t]) for t in range(T)]
            rho = [min(rho_bar, x) for x in ratio]
            cc = [lam * min(c_bar, x) for x in ratio]
            for s in range(T):
                k = _episode_end(term, trunc, s, T)
                edge = _edge_value(k, T, term, trunc, d["tv"][e], d["b"][e])
                total = 0.0
                for t in range(s, k + 1):
                    nxt = d["v"][e, t + 1] if t < k else edge
                    delta = rho[t] * (d["r"][e, t] + g * nxt - d["v"][e, t])
                    total += g ** (t - s) * np.prod(cc[s:t]) * delta
                wvs[e, s] = d["v"][e, s] + total
            for s in range(T):
                k = _episode_end(term, trunc, s, T)
                edge = _edge_value(k, T, term, trunc, d["tv"][e], d["b"][e])
                nvs = wvs[e, s + 1] if s < k else edge
                wpg[e, s] = rho[s] * (d["r"][e, s] + g * nvs - d["v"][e, s])
        _close(vs, wvs, what=f"V-Trace vs brute force T={T}")
        _close(pg, wpg, what=f"V-Trace pg brute force T={T}")


def pin_vtrace_on_policy(ref):
    """pi = mu, rho_bar = c_bar = 1: vs is the bootstrapped discounted
    return and pg_adv is that return minus the value."""
    rng = np.random.default_rng(19)
    d = _vtrace_inputs(rng, 6, 13)
    vs, pg = ref.vtrace(d["r"], d["v"], d["lp"], d["lp"], d["term"], d["trunc"], d["tv"], d["b"],
                        gamma=0.96)
    G = ref.discounted_return(d["r"], d["term"], d["trunc"], d["tv"], d["b"], gamma=0.96)
    _close(vs, G, what="V-Trace on-policy vs")
    _close(pg, G - d["v"], what="V-Trace on-policy pg")


# --------------------------------------------------------------------------
# Retrace(lambda)
# --------------------------------------------------------------------------

def _retrace_inputs(rng, E, T, A=4):
    d = _random_rollout(rng, E, T)
    d["q"] = rng.normal(size=(E, T, A))
    p = rng.random((E, T, A)) + 0.05
    d["pi"] = p / p.sum(-1, keepdims=True)
    d["a"] = rng.integers(0, A, size=(E, T)).astype(np.int32)
    d["mu_a"] = rng.uniform(0.05, 0.9, size=(E, T))
    return d


def _retrace_call(ref, d, g, lam):
    return ref.retrace(d["q"], d["pi"], d["mu_a"], d["a"], d["r"], d["term"], d["trunc"], d["tv"],
                       d["b"], gamma=g, lam=lam)


def pin_retrace_bruteforce(ref):
    """Q^ret_t = Q(x_t,a_t) + sum_{s=t}^{end} g^(s-t) (prod_{i=t+1}^{s} c_i)
    delta_s, delta_s = r_s + g * next_s - Q(x_s,a_s), next_s = E_pi Q(x_{s+1})
    inside the stretch and the edge value at its end."""
    rng = np.random.default_rng(20)
    g, lam = 0.9, 0.85
    for T in (1, 2, 3, 6):
        d = _retrace_inputs(rng, 5, T)
        got = _retrace_call(ref, d, g, lam)
        want = np.zeros_like(got)
        A = d["q"].shape[-1]
        for e in range(5):
            term, trunc = d["term"][e], d["trunc"][e]
            ev = [sum(d["pi"][e, t, a] * d["q"][e, t, a] for a in range(A)) for t in range(T)]
            qa = [d["q"][e, t, d["a"][e, t]] for t in range(T)]
            cc = [lam * min(1.0, d["pi"][e, t, d["a"][e, t]] / d["mu_a"][e, t]) for t in range(T)]
            for t in range(T):
                k = _episode_end(term, trunc, t, T)
                edge = _edge_value(k, T, term, trunc, d["tv"][e], d["b"][e])
                total = 0.0
                for s in range(t, k + 1):
                    nxt = ev[s + 1] if s < k else edge
                    delta = d["r"][e, s] + g * nxt - qa[s]
                    total += g ** (s - t) * np.prod(cc[t + 1:s + 1]) * delta
                want[e, t] = qa[t] + total
        _close(got, want, what=f"Retrace brute force T={T}")


def pin_retrace_lambda0(ref):
    """lam = 0: the target is the expected-SARSA one-step target
    r_t + g * E_pi Q(x_{t+1}) (edge value at a stretch end)."""
    rng = np.random.default_rng(21)
    g = 0.95
    d = _retrace_inputs(rng, 5, 8)
    got = _retrace_call(ref, d, g, 0.0)
    want = np.zeros_like(got)
    E, T, A = d["q"].shape
    for e in range(E):
        term, trunc = d["term"][e], d["trunc"][e]
        for t in range(T):
            k = _episode_end(term, trunc, t, T)
            if t < k:
                nxt = sum(d["pi"][e, t + 1, a] * d["q"][e, t + 1, a] for a in range(A))
            else:
                nxt = _edge_value(k, T, term, trunc, d["tv"][e], d["b"][e])
            want[e, t] = d["r"][e, t] + g * nxt
    _close(got, want, what="Retrace lam=0")


def pin_retrace_on_policy_constant_q(ref):
    """lam = 1, mu = pi on the taken action, Q constant over actions: the
    traces are 1 and the target is the bootstrapped discounted return."""
    rng = np.random.default_rng(22)
    d = _retrace_inputs(rng, 5, 10)
    d["q"] = np.repeat(rng.normal(size=(5, 10, 1)), d["q"].shape[-1], axis=-1)
    d["mu_a"] = np.take_along_axis(d["pi"], d["a"][..., None].astype(np.int64), -1)[..., 0]
    got = _retrace_call(ref, d, 0.93, 1.0)
    G = ref.discounted_return(d["r"], d["term"], d["trunc"], d["tv"], d["b"], gamma=0.93)
    _close(got, G, what="Retrace on-policy constant Q")


# --------------------------------------------------------------------------
# forward scans
# --------------------------------------------------------------------------

def _stretch_start(done, t, flag_is_start=False):
    """First step of t's episode: after the last flagged step before t
    (flag = last step), or at the last flagged step <= t (flag = first)."""
    s = t
    if flag_is_start:
        while s > 0 and not done[s]:
            s -= 1
    else:
        while s > 0 and not done[s - 1]:
            s -= 1
    return s


def pin_elig_closed_form(ref):
    """x = 1, no boundaries: e_t = (1 - (g*lam)^(t+1)) / (1 - g*lam)."""
    E, T, g, lam = 2, 40, 0.99, 0.9
    got = ref.eligibility_trace(np.ones((E, T)), np.zeros((E, T), np.uint8), gamma=g, lam=lam)
    t = np.arange(T)
    want = np.broadcast_to((1 - (g * lam) ** (t + 1)) / (1 - g * lam), (E, T))
    _close(got, want, what="eligibility closed form")


def pin_elig_bruteforce(ref):
    rng = np.random.default_rng(23)
    g, lam = 0.9, 0.8
    for T in (1, 2, 5, 7):
        d = _random_rollout(rng, 5, T)
        x = rng.normal(size=(5, T))
        got = ref.eligibility_trace(x, d["term"], d["trunc"], gamma=g, lam=lam)
        want = np.zeros_like(got)
        for e in range(5):
            done = (d["term"][e] | d["trunc"][e]) != 0
            for t in range(T):
                s0 = _stretch_start(done, t)
                want[e, t] = sum((g * lam) ** (t - s) * x[e, s] for s in range(s0, t + 1))
        _close(got, want, what=f"eligibility brute force T={T}")


def pin_prefix_sum_counter(ref):
    """x = 1: the inclusive sum counts the steps of the episode so far."""
    T = 12
    term = np.zeros((1, T), np.uint8)
    term[0, [3, 4, 9]] = 1
    got = ref.episodic_prefix_sum(np.ones((1, T), np.int32), term)
    want = np.array([[1, 2, 3, 4, 1, 1, 2, 3, 4, 5, 1, 2]])
    assert np.array_equal(got, want), got
    got_x = ref.episodic_prefix_sum(np.ones((1, T), np.int32), term, exclusive=True)
    assert np.array_equal(got_x, want - 1), got_x
    got_s = ref.episodic_prefix_sum(np.ones((1, T), np.int32), term, flag_is_start=True)
    want_s = np.array([[1, 2, 3, 1, 1, 2, 3, 4, 5, 1, 2, 3]])
    assert np.array_equal(got_s, want_s), got_s


def pin_prefix_sum_bruteforce(ref):
    rng = np.random.default_rng(24)
    for T in (1, 3, 8):
        d = _random_rollout(rng, 6, T, p_term=0.25, p_trunc=0.15)
        xi = rng.integers(-50, 50, size=(6, T)).astype(np.int32)
        xf = rng.normal(size=(6, T))
        for flag_is_start in (False, True):
            for exclusive in (False, True):
                gi = ref.episodic_prefix_sum(xi, d["term"], d["trunc"], exclusive, flag_is_start)
                gf = ref.episodic_prefix_sum(xf, d["term"], d["trunc"], exclusive, flag_is_start)
                wi = np.zeros((6, T), np.int64)
                wf = np.zeros((6, T))
                for e in range(6):
                    done = (d["term"][e] | d["trunc"][e]) != 0
                    for t in range(T):
                        s0 = _stretch_start(done, t, flag_is_start)
                        stop = t if exclusive else t + 1
                        wi[e, t] = sum(int(xi[e, s]) for s in range(s0, stop))
                        wf[e, t] = sum(xf[e, s] for s in range(s0, stop))
                assert gi.dtype == np.int32 and np.array_equal(gi, wi), (flag_is_start, exclusive)
                _close(gf, wf, what=f"prefix sum f T={T}")


def pin_prefix_sum_int32_wraps(ref):
    """int32 sums wrap modulo 2^32 (two's complement)."""
    x = np.array([[2 ** 31 - 1, 2 ** 31 - 1, 5, -7]], np.int32)
    got = ref.episodic_prefix_sum(x, np.zeros((1, 4), np.uint8))
    want = np.array([[2 ** 31 - 1, -2, 3, -4]], np.int32)
    assert np.array_equal(got, want), got


# --------------------------------------------------------------------------
# no-leak invariant (§5 Correctness Analysis)
# --------------------------------------------------------------------------

def pin_no_leak(ref):
    """Perturbing every input strictly after a boundary at t* leaves the
    backward estimators' outputs at t <= t* bit-identical (for a truncation
    the continuation value at t* itself is kept); perturbing every input at
    or before t* leaves the forward scans' outputs after t* bit-identical."""
    rng = np.random.default_rng(25)
    E, T, ts = 4, 12, 5
    for kind in ("term", "trunc"):
        d = _retrace_inputs(rng, E, T)
        d["lp"] = rng.normal(size=(E, T))
        d["lm"] = rng.normal(size=(E, T))
        d["term"][:, ts] = 1 if kind == "term" else 0
        d["trunc"][:, ts] = 1 if kind == "trunc" else 0
        p = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in d.items()}
        after = slice(ts + 1, None)
        for key in ("r", "v", "tv", "lp", "lm"):
            p[key][:, after] = rng.normal(size=p[key][:, after].shape) + 3.0
        p["mu_a"][:, after] = rng.uniform(0.05, 0.9, size=p["mu_a"][:, after].shape)
        p["pi"][:, after] = p["pi"][:, after][..., ::-1]
        p["q"][:, after] = rng.normal(size=p["q"][:, after].shape)
        p["a"][:, after] = (p["a"][:, after] + 1) % p["q"].shape[-1]
        p["term"][:, after] = rng.random((E, T - ts - 1)) < 0.3
        p["trunc"][:, after] = rng.random((E, T - ts - 1)) < 0.3
        p["b"] = p["b"] + 1.0

        def run(x):
            return [
                *ref.gae(x["r"], x["v"], x["term"], x["trunc"], x["tv"], x["b"]),
                ref.discounted_return(x["r"], x["term"], x["trunc"], x["tv"], x["b"]),
                ref.td_lambda(x["r"], x["v"], x["term"], x["trunc"], x["tv"], x["b"]),
                *ref.vtrace(x["r"], x["v"], x["lp"], x["lm"], x["term"], x["trunc"], x["tv"], x["b"]),
                _retrace_call(ref, x, 0.99, 0.95),
            ]
        for a, b in zip(run(d), run(p)):
            assert np.array_equal(a[:, :ts + 1], b[:, :ts + 1]), f"backward leak across {kind}"

    d = _random_rollout(rng, E, T)
    d["term"][:, ts] = 1
    x = rng.normal(size=(E, T))
    xi = rng.integers(0, 9, size=(E, T)).astype(np.int32)
    p = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in d.items()}
    px, pxi = x.copy(), xi.copy()
    before = slice(0, ts)
    px[:, :ts + 1] += 2.0
    pxi[:, :ts + 1] += 3
    p["term"][:, before] = rng.random((E, ts)) < 0.4
    p["trunc"][:, before] = rng.random((E, ts)) < 0.4
    pairs = [
        (ref.eligibility_trace(x, d["term"], d["trunc"]), ref.eligibility_trace(px, p["term"], p["trunc"])),
        (ref.episodic_prefix_sum(xi, d["term"], d["trunc"]),
         ref.episodic_prefix_sum(pxi, p["term"], p["trunc"])),
        (ref.episodic_prefix_sum(x, d["term"], d["trunc"], exclusive=True),
         ref.episodic_prefix_sum(px, p["term"], p["trunc"], exclusive=True)),
    ]
    for a, b in pairs:
        assert np.array_equal(a[:, ts + 1:], b[:, ts + 1:]), "forward leak across boundary"


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

"""Float64 sequential reference of the seven credit-assignment estimators.

TEST INFRASTRUCTURE: only the test suite, the smoke check and the
benchmark's CPU-baseline leg use this module.  It shares no code with the
CUDA path.

Source: "rl-triton: High-Performance Triton GPU Kernels for Reinforcement
Learning Credit Assignment" (arXiv:2608.17641), §1 Introduction and §3 The
Unified Linear Recurrence Framework, with the per-estimator definitions of
the primary works that paper cites: GAE [Schulman et al., 2016], V-Trace
[Espeholt et al., 2018] and Retrace(lambda) [Munos et al., 2016].

Every estimator here is written as its plain time-step loop, NOT as the
(alpha, beta) affine scan that the kernels evaluate: the loop runs from the
last step backwards (GAE, V-Trace, Retrace, TD(lambda), discounted return)
or from the first step forwards (eligibility trace, episodic prefix sum),
in float64, vectorised only across the independent environment rows.  The
only scan-shaped function is :func:`affine_scan`, the sequential definition
of the recurrence A_t = alpha_t + beta_t * A_{t+1} itself (§2.2 Associative
Scan), which the generic kernel entry point evaluates.

Layout: every rollout array is env-major ``[E, T]`` (per-action arrays
``[E, T, A]``), per-environment vectors ``[E]``.  Inputs of any float type
are converted to float64 exactly; outputs are float64 (int32 for the integer
prefix sum).

Episode-boundary rules (§3.2 Episode-boundary semantics), one reading where
the pages are silent marked READING:
  * ``terminated[e, t] != 0``: the episode ended at t; the successor value is
    0 and nothing from t+1 on flows into t.
  * ``truncated[e, t] != 0``: the episode was cut at t; the successor value
    is the caller's continuation value ``trunc_value[e, t]`` and nothing
    from t+1 on flows into t.  READING: where both flags are set,
    termination wins; ``trunc_value`` is a dense [E, T] tensor read only at
    truncated steps.
  * t = T-1 with neither flag: the rollout window ends; the successor value
    is ``bootstrap[e]`` (0 if ``bootstrap`` is None).
  * the forward scans (eligibility trace, prefix sum) restart after a step
    whose flag is set and take no bootstrap at all (§5 Correctness Analysis,
    episode boundaries of the forward scans).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "affine_scan", "gae", "discounted_return", "td_lambda", "vtrace",
    "retrace", "eligibility_trace", "episodic_prefix_sum",
]


# --------------------------------------------------------------------------
# input handling (no arithmetic of the method)
# --------------------------------------------------------------------------

def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def _flag(a, E, T):
    if a is None:
        return np.zeros((E, T), dtype=bool)
    a = np.asarray(a)
    assert a.shape == (E, T), (a.shape, (E, T))
    return a != 0


def _boundaries(terminated, truncated, trunc_value, E, T):
    """(term, trunc, trunc_value) with truncation cleared where the step
    also terminates (READING: termination wins)."""
    term = _flag(terminated, E, T)
    trunc = _flag(truncated, E, T) & ~term
    if truncated is not None and trunc_value is None:
        raise ValueError("truncated given without trunc_value")
    tv = _f64(trunc_value) if trunc_value is not None else np.zeros((E, T))
    return term, trunc, tv


def _bootstrap(bootstrap, E):
    return np.zeros(E) if bootstrap is None else _f64(bootstrap).reshape(E)


def _successor(t, T, interior, term, trunc, tv, boot):
    """Value that step t bootstraps from (§3.2): 0 after a termination, the
    caller's continuation value after a truncation, the window bootstrap at
    t = T-1, else ``interior`` (the continuation through step t+1)."""
    nxt = boot if t == T - 1 else interior
    nxt = np.where(trunc[:, t], tv[:, t], nxt)
    return np.where(term[:, t], 0.0, nxt)


def _continues(t, T, term, trunc):
    """True where step t's result depends on step t+1's (no episode boundary
    at t and t is not the last step of the window)."""
    return ~(term[:, t] | trunc[:, t]) & (t < T - 1)


# --------------------------------------------------------------------------
# the recurrence itself
# --------------------------------------------------------------------------

def affine_scan(alpha, beta, carry=None, reverse=True):
    """Sequential first-order linear recurrence (§1 Introduction, §2.2).

    reverse=True:  A_t = alpha_t + beta_t * A_{t+1},  A_T = carry.
    reverse=False: A_t = alpha_t + beta_t * A_{t-1},  A_{-1} = carry.
    ``carry`` is [E] (0 where None).  Returns A [E, T] float64.
    """
    a, b = _f64(alpha), _f64(beta)
    E, T = a.shape
    A = np.zeros(E) if carry is None else _f64(carry).reshape(E).copy()
    out = np.empty((E, T))
    steps = range(T - 1, -1, -1) if reverse else range(T)
    for t in steps:
        A = a[:, t] + b[:, t] * A
        out[:, t] = A
    return out


# --------------------------------------------------------------------------
# backward estimators
# --------------------------------------------------------------------------

def gae(rewards, values, terminated, truncated=None, trunc_value=None,
        bootstrap=None, gamma=0.99, lam=0.95):
    """Generalized Advantage Estimation [Schulman et al., 2016] (§2.1
    Motivation: each advantage depends on the next one).

        delta_t = r_t + gamma * V_next(t) - V_t
        A_t     = delta_t + gamma * lam * A_{t+1}   (only while the episode
                                                     continues inside the
                                                     window)
        R_t     = A_t + V_t

    V_next(t) follows the boundary rules of the module docstring; the window
    bootstrap enters delta_{T-1} locally (§3.2).  Returns (adv, ret).
    """
    r, v = _f64(rewards), _f64(values)
    E, T = r.shape
    term, trunc, tv = _boundaries(terminated, truncated, trunc_value, E, T)
    boot = _bootstrap(bootstrap, E)
    adv = np.empty((E, T))
    later = np.zeros(E)                       # A_{t+1}
    for t in range(T - 1, -1, -1):
        v_next = v[:, t + 1] if t + 1 < T else None
        delta = r[:, t] + gamma * _successor(t, T, v_next, term, trunc, tv, boot) - v[:, t]
        adv[:, t] = delta + gamma * lam * np.where(_continues(t, T, term, trunc), later, 0.0)
        later = adv[:, t]
    return adv, adv + v


def discounted_return(rewards, terminated, truncated=None, trunc_value=None,
                      bootstrap=None, gamma=0.99):
    """Discounted return G_t = r_t + gamma * G_next(t), where G_next(t) is
    G_{t+1} inside an episode and the boundary value (0 / continuation value
    / window bootstrap) at its edge (§3.2)."""
    r = _f64(rewards)
    E, T = r.shape
    term, trunc, tv = _boundaries(terminated, truncated, trunc_value, E, T)
    boot = _bootstrap(bootstrap, E)
    ret = np.empty((E, T))
    later = None                              # G_{t+1}
    for t in range(T - 1, -1, -1):
        ret[:, t] = r[:, t] + gamma * _successor(t, T, later, term, trunc, tv, boot)
        later = ret[:, t]
    return ret


def td_lambda(rewards, values, terminated, truncated=None, trunc_value=None,
              bootstrap=None, gamma=0.99, lam=0.95):
    """TD(lambda) return in its recursive form:

        G_t = r_t + gamma * [(1 - lam) * V_{t+1} + lam * G_{t+1}]

    inside an episode; at an episode or window edge the bracket is the
    boundary value (0 / continuation value / window bootstrap) (§3.2)."""
    r, v = _f64(rewards), _f64(values)
    E, T = r.shape
    term, trunc, tv = _boundaries(terminated, truncated, trunc_value, E, T)
    boot = _bootstrap(bootstrap, E)
    ret = np.empty((E, T))
    later = None                              # G_{t+1}
    for t in range(T - 1, -1, -1):
        interior = None if t == T - 1 else (1.0 - lam) * v[:, t + 1] + lam * later
        ret[:, t] = r[:, t] + gamma * _successor(t, T, interior, term, trunc, tv, boot)
        later = ret[:, t]
    return ret


def vtrace(rewards, values, logp_target, logp_behaviour, terminated,
           truncated=None, trunc_value=None, bootstrap=None, gamma=0.99,
           rho_bar=1.0, c_bar=1.0, lam=1.0):
    """V-Trace targets and policy-gradient advantages [Espeholt et al., 2018]
    (§8 Related Work, off-policy correction).

        ratio_t = exp(logp_target_t - logp_behaviour_t)
        rho_t   = min(rho_bar, ratio_t)
        c_t     = lam * min(c_bar, ratio_t)
        delta_t = rho_t * (r_t + gamma * V_next(t) - V_t)
        vs_t - V_t = delta_t + gamma * c_t * (vs_{t+1} - V_{t+1})
                     (only while the episode continues inside the window)
        pg_adv_t = rho_t * (r_t + gamma * vs_next(t) - V_t)

    V_next(t) follows the boundary rules; vs_next(t) is the same with vs_{t+1}
    in place of V_{t+1}.  READING: the policy-gradient clip uses rho_bar;
    lam defaults to 1 (plain V-Trace).  Returns (vs, pg_adv).
    """
    r, v = _f64(rewards), _f64(values)
    E, T = r.shape
    term, trunc, tv = _boundaries(terminated, truncated, trunc_value, E, T)
    boot = _bootstrap(bootstrap, E)
    ratio = np.exp(_f64(logp_target) - _f64(logp_behaviour))
    rho = np.minimum(rho_bar, ratio)
    c = lam * np.minimum(c_bar, ratio)
    vs = np.empty((E, T))
    pg = np.empty((E, T))
    later_gap = np.zeros(E)                   # vs_{t+1} - V_{t+1}
    later_vs = None                           # vs_{t+1}
    for t in range(T - 1, -1, -1):
        v_next = v[:, t + 1] if t + 1 < T else None
        delta = rho[:, t] * (r[:, t] + gamma * _successor(t, T, v_next, term, trunc, tv, boot) - v[:, t])
        gap = delta + gamma * c[:, t] * np.where(_continues(t, T, term, trunc), later_gap, 0.0)
        vs[:, t] = v[:, t] + gap
        pg[:, t] = rho[:, t] * (r[:, t] + gamma * _successor(t, T, later_vs, term, trunc, tv, boot) - v[:, t])
        later_gap = gap
        later_vs = vs[:, t]
    return vs, pg


def retrace(q, pi, mu_a, actions, rewards, terminated, truncated=None,
            trunc_value=None, bootstrap=None, gamma=0.99, lam=0.95):
    """Retrace(lambda) Q targets [Munos et al., 2016] (§3.3: the decay sits on
    the next step's importance weight).

        EV_t  = sum_a pi(a | x_t) * Q(x_t, a)
        c_t   = lam * min(1, pi(a_t | x_t) / mu(a_t | x_t))
        G_t   = r_t + gamma * [EV_{t+1} + c_{t+1} * (G_{t+1} - Q(x_{t+1}, a_{t+1}))]

    inside an episode; at an edge the bracket is the boundary value: 0 after
    a termination, ``trunc_value`` (E_pi Q of the truncated episode's last
    state) after a truncation, ``bootstrap`` (E_pi Q of the state after the
    window) at t = T-1.  q, pi: [E, T, A]; mu_a: behaviour probability of the
    taken action [E, T] (must be > 0); actions: [E, T] ints in [0, A).
    """
    Q, P = _f64(q), _f64(pi)
    r = _f64(rewards)
    E, T, A = Q.shape
    a = np.asarray(actions).astype(np.int64)[..., None]
    term, trunc, tv = _boundaries(terminated, truncated, trunc_value, E, T)
    boot = _bootstrap(bootstrap, E)
    ev = np.sum(P * Q, axis=-1)
    q_taken = np.take_along_axis(Q, a, axis=-1)[..., 0]
    p_taken = np.take_along_axis(P, a, axis=-1)[..., 0]
    with np.errstate(divide="ignore"):
        c = lam * np.minimum(1.0, p_taken / _f64(mu_a))
    out = np.empty((E, T))
    later = None                              # G_{t+1}
    for t in range(T - 1, -1, -1):
        interior = None if t == T - 1 else ev[:, t + 1] + c[:, t + 1] * (later - q_taken[:, t + 1])
        out[:, t] = r[:, t] + gamma * _successor(t, T, interior, term, trunc, tv, boot)
        later = out[:, t]
    return out


# --------------------------------------------------------------------------
# forward estimators
# --------------------------------------------------------------------------

def eligibility_trace(x, terminated, truncated=None, gamma=0.99, lam=0.95):
    """Accumulating eligibility trace, run forward in time (§1, forward-time
    mirror; §5, forward-scan boundaries):

        e_t = x_t + gamma * lam * e_{t-1},   restarting at e_t = x_t on the
                                             first step of a rollout and on
                                             every step after a flagged one.

    READING: x_t is the caller's per-step signal (x = 1 counts visits)."""
    xs = _f64(x)
    E, T = xs.shape
    done = _flag(terminated, E, T) | _flag(truncated, E, T)
    out = np.empty((E, T))
    prev = np.zeros(E)
    for t in range(T):
        starts = np.ones(E, bool) if t == 0 else done[:, t - 1]
        prev = xs[:, t] + gamma * lam * np.where(starts, 0.0, prev)
        out[:, t] = prev
    return out


def episodic_prefix_sum(x, terminated, truncated=None, exclusive=False,
                        flag_is_start=False):
    """Running sum of x within each episode, forward in time (§3.3: segmented
    forward scan with configurable boundary conventions).

    READING of the conventions:
      * inclusive (default): S_t = sum of x over the steps of t's episode up
        to and including t; exclusive: the same sum over the steps before t.
      * default boundary: a flagged step (terminated or truncated) is the
        LAST step of its episode; ``flag_is_start``: a flagged step is the
        FIRST step of a new episode.
      * integer x is summed in int32 with two's-complement wraparound; float
        x in float64.
    """
    xv = np.asarray(x)
    E, T = xv.shape
    integer = np.issubdtype(xv.dtype, np.integer)
    if integer:
        xs = xv.astype(np.int64) & 0xFFFFFFFF      # the uint32 bit pattern
    else:
        xs = xv.astype(np.float64)
    flag = _flag(terminated, E, T) | _flag(truncated, E, T)
    out = np.empty((E, T), dtype=np.int64 if integer else np.float64)
    running = np.zeros(E, dtype=xs.dtype)           # inclusive sum at t-1
    for t in range(T):
        if flag_is_start:
            starts = np.ones(E, bool) if t == 0 else flag[:, t]
        else:
            starts = np.ones(E, bool) if t == 0 else flag[:, t - 1]
        before = np.where(starts, 0, running)
        running = before + xs[:, t]
        if integer:
            running = running & 0xFFFFFFFF
        out[:, t] = before if exclusive else running
    if integer:
        return out.astype(np.uint32).view(np.int32)
    return out

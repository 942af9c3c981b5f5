"""Seeded synthetic rollouts for the credit-assignment scans.

This module only draws inputs: it holds none of the estimators' arithmetic,
so the CUDA path and the float64 oracle can both be fed from it without
sharing any computation.  Every draw comes from one ``torch.Generator``
(on the device the arrays are made on) seeded per workload, in a fixed
order, so a seed and a device type fix the inputs bit for bit.

The workloads follow the shapes and distributions of the rl-triton paper
(arXiv:2608.17641) benchmarks, "massively parallel simulation regime"
(thousands of environments, short rollouts; §6 Benchmarking Methodology,
§7 Results): float32 rewards and values drawn N(0, 1), Bernoulli
termination and truncation flags (disjoint), a per-environment bootstrap
value for the rollout-window edge, and a dense truncation-value tensor that
is only read where a step is truncated.  The policy inputs of V-Trace and
Retrace(lambda) come from 18-action softmax / log-softmax of N(0, 1) logits.

Arrays are torch tensors on the requested device (CPU by default),
env-major ``[E, T]`` (``[E, T, A]`` for per-action tensors);
:func:`to_time_major` re-lays them out as ``[T, E]`` and :func:`numpy`
turns a dict of them into numpy arrays.
"""
from __future__ import annotations

import zlib

import numpy as np
import torch

NUM_ACTIONS = 18


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _flags(g: torch.Generator, E: int, T: int, p_term: float, p_trunc: float):
    """Termination then truncation flags as uint8, truncation cleared where
    the step also terminates (the two are drawn disjoint)."""
    dev = g.device
    term = torch.rand(E, T, generator=g, device=dev) < p_term
    trunc = (torch.rand(E, T, generator=g, device=dev) < p_trunc) & ~term
    return term.to(torch.uint8), trunc.to(torch.uint8)


def numpy(d: dict) -> dict:
    """The same dict with every tensor as a CPU numpy array."""
    return {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def config_seed(name: str) -> int:
    """Stable per-workload seed (crc32 of the workload's name)."""
    return zlib.crc32(name.encode()) & 0x7FFFFFFF


def value_rollout(E: int, T: int, seed: int, p_term: float = 0.05, p_trunc: float = 0.02,
                  with_trunc: bool = True, device="cpu") -> dict:
    """Inputs of GAE, TD(lambda) and discounted returns.

    Draw order: rewards [E,T], values [E,T], bootstrap [E], trunc_value
    [E,T], termination flags, truncation flags.  With ``with_trunc=False``
    the truncation flags are still drawn (so the other arrays do not move)
    but returned as ``None``.
    """
    g = _gen(seed, device)
    rewards = torch.randn(E, T, generator=g, device=device)
    values = torch.randn(E, T, generator=g, device=device)
    bootstrap = torch.randn(E, generator=g, device=device)
    trunc_value = torch.randn(E, T, generator=g, device=device)
    term, trunc = _flags(g, E, T, p_term, p_trunc)
    return dict(rewards=rewards, values=values, bootstrap=bootstrap,
                trunc_value=trunc_value if with_trunc else None,
                terminated=term, truncated=trunc if with_trunc else None)


def vtrace_rollout(E: int, T: int, seed: int, p_term: float = 0.01, p_trunc: float = 0.0,
                   with_trunc: bool = False, num_actions: int = NUM_ACTIONS, device="cpu") -> dict:
    """Inputs of V-Trace.

    Target and behaviour logits are N(0,1) over ``num_actions``; the taken
    action is sampled from the behaviour policy; the log-probabilities of the
    taken action under both policies are returned (the kernel's inputs).
    Draw order: rewards, values, bootstrap, trunc_value, target logits,
    behaviour logits, sampled actions, flags.
    """
    g = _gen(seed, device)
    rewards = torch.randn(E, T, generator=g, device=device)
    values = torch.randn(E, T, generator=g, device=device)
    bootstrap = torch.randn(E, generator=g, device=device)
    trunc_value = torch.randn(E, T, generator=g, device=device)
    logits_pi = torch.randn(E, T, num_actions, generator=g, device=device)
    logits_mu = torch.randn(E, T, num_actions, generator=g, device=device)
    logp_pi = torch.log_softmax(logits_pi, dim=-1)
    logp_mu = torch.log_softmax(logits_mu, dim=-1)
    # the taken action is sampled from the behaviour policy
    flat = logp_mu.exp().reshape(E * T, num_actions)
    actions = torch.multinomial(flat, 1, generator=g).reshape(E, T, 1)
    lp_pi = torch.gather(logp_pi, -1, actions).squeeze(-1)
    lp_mu = torch.gather(logp_mu, -1, actions).squeeze(-1)
    term, trunc = _flags(g, E, T, p_term, p_trunc)
    return dict(rewards=rewards, values=values, bootstrap=bootstrap,
                trunc_value=trunc_value if with_trunc else None,
                logp_target=lp_pi.contiguous(), logp_behaviour=lp_mu.contiguous(),
                actions=actions.squeeze(-1).to(torch.int32),
                terminated=term, truncated=trunc if with_trunc else None)


def retrace_rollout(E: int, T: int, seed: int, p_term: float = 0.002, p_trunc: float = 0.0,
                    with_trunc: bool = False, num_actions: int = NUM_ACTIONS, device="cpu") -> dict:
    """Inputs of Retrace(lambda).

    Q [E,T,A] ~ N(0,1); target policy pi = softmax(N(0,1) logits) [E,T,A];
    behaviour policy mu = softmax(N(0,1) logits), of which only the taken
    action's probability mu_a [E,T] is passed on; actions uniform in [0, A).
    bootstrap [E] ~ N(0,1) stands for E_pi Q at the state after the window.
    Draw order: rewards, Q, target logits, behaviour logits, actions,
    bootstrap, trunc_value, flags.
    """
    g = _gen(seed, device)
    rewards = torch.randn(E, T, generator=g, device=device)
    q = torch.randn(E, T, num_actions, generator=g, device=device)
    pi = torch.softmax(torch.randn(E, T, num_actions, generator=g, device=device), dim=-1)
    mu = torch.softmax(torch.randn(E, T, num_actions, generator=g, device=device), dim=-1)
    actions = torch.randint(0, num_actions, (E, T), generator=g, device=device)
    bootstrap = torch.randn(E, generator=g, device=device)
    trunc_value = torch.randn(E, T, generator=g, device=device)
    mu_a = torch.gather(mu, -1, actions.unsqueeze(-1)).squeeze(-1)
    term, trunc = _flags(g, E, T, p_term, p_trunc)
    return dict(rewards=rewards, q=q, pi=pi, mu_a=mu_a.contiguous(),
                actions=actions.to(torch.int32), bootstrap=bootstrap,
                trunc_value=trunc_value if with_trunc else None,
                terminated=term, truncated=trunc if with_trunc else None)


def forward_rollout(E: int, T: int, seed: int, p_term: float = 0.01, p_trunc: float = 0.005,
                    with_trunc: bool = True, int_max: int = 16, device="cpu") -> dict:
    """Inputs of the forward scans (eligibility traces, episodic prefix sums).

    x_f32 [E,T] ~ N(0,1) (trace signal / float prefix-sum input) and
    x_i32 [E,T] ~ U{0, ..., int_max-1}.  Draw order: x_f32, x_i32, flags.
    """
    g = _gen(seed, device)
    x_f32 = torch.randn(E, T, generator=g, device=device)
    x_i32 = torch.randint(0, int_max, (E, T), generator=g, device=device).to(torch.int32)
    term, trunc = _flags(g, E, T, p_term, p_trunc)
    return dict(x_f32=x_f32, x_i32=x_i32, terminated=term,
                truncated=trunc if with_trunc else None)


def affine_rollout(E: int, T: int, seed: int, beta_lo: float = -1.0, beta_hi: float = 1.0,
                   device="cpu") -> dict:
    """Inputs of the generic scan: alpha ~ N(0,1), beta ~ U(beta_lo, beta_hi),
    carry [E] ~ N(0,1); about 2% of the betas are exactly zero (resets)."""
    g = _gen(seed, device)
    alpha = torch.randn(E, T, generator=g, device=device)
    beta = beta_lo + (beta_hi - beta_lo) * torch.rand(E, T, generator=g, device=device)
    zero = torch.rand(E, T, generator=g, device=device) < 0.02
    beta = torch.where(zero, torch.zeros_like(beta), beta)
    carry = torch.randn(E, generator=g, device=device)
    return dict(alpha=alpha, beta=beta, carry=carry)


def to_time_major(a):
    """[E, T] -> [T, E] and [E, T, A] -> [T, E, A] (contiguous, numpy or
    torch); None and per-environment [E] vectors pass through unchanged."""
    if a is None or a.ndim == 1:
        return a
    if isinstance(a, torch.Tensor):
        return a.transpose(0, 1).contiguous()
    if a.ndim == 2:
        return np.ascontiguousarray(a.T)
    return np.ascontiguousarray(a.transpose(1, 0, 2))


def from_time_major(a):
    """Inverse of :func:`to_time_major`."""
    return to_time_major(a)

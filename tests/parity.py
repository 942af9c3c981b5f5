"""Parity harness: the CUDA path (through the C ABI) against the float64
oracle on the same seeded inputs.

Floating-point outputs must satisfy max |gpu - ref| / (1 + |ref|) <= 1e-4
(the bar rl-triton's §6 validation applies before timing, atol = rtol =
1e-4, written as one combined bound); int32 outputs must be bit-exact.
Large cases compare a sample of whole rows (rows are independent, so the
oracle can evaluate any row on its own), always including the first and
last row.
"""
from __future__ import annotations

import numpy as np
import torch

from first_order_linear_gb300 import rlca, synth
from oracle import rlca_ref as ref

TOL = 1e-4
GAMMA, LAMBDA = 0.99, 0.95


# bfloat16 outputs (RLCA_BF16): the float32 result, within TOL of the
# oracle, is rounded to nearest once.  A bfloat16 keeps 8 significant bits,
# so rounding moves x by at most half an ulp <= 2^-8 |x|; with |x - ref| <=
# TOL (1 + |ref|) that gives |out - ref| <= 2^-8 |ref| + TOL (1 + 2^-8) (1 + |ref|).
BF16_REL = 2.0 ** -8
BF16_TOL = TOL * (1.0 + 2.0 ** -8)


def assert_close(got, want, what, tol=TOL, rel=0.0):
    """max |got - want| <= tol (1 + |want|) + rel |want| (bit-exact for ints);
    returns the worst |got - want| / (tol (1 + |want|) + rel |want|) * tol."""
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if np.issubdtype(want.dtype, np.integer):
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{what}: {len(bad)} int mismatches, first at {bad[:3].tolist()}"
        return 0.0
    g = got.astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    bound = tol * (1.0 + np.abs(want)) + rel * np.abs(want)
    err = tol * np.abs(g - want) / bound
    worst = float(err.max()) if err.size else 0.0
    if worst > tol:
        idx = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(f"{what}: error {worst / tol:.3f} x the bound at {idx}: gpu {g[idx]!r} ref {want[idx]!r}")
    return worst


def sample_rows(E, T, seed, limit=1 << 20, n=96):
    if E * T <= limit:
        return np.arange(E)
    rng = np.random.default_rng(seed)
    rows = rng.choice(E, size=min(n, E), replace=False)
    return np.unique(np.concatenate([rows, [0, E - 1]]))


def _np(t, rows=None):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:  # exact in float32
        t = t.float()
    if rows is None or t.dim() == 0:
        return t.cpu().numpy()
    return t[torch.as_tensor(rows, device=t.device)].cpu().numpy()


def to_bf16(d):
    """The float32 tensors of an input dict rounded to bfloat16 (the values
    both sides then take as exact inputs)."""
    return {k: (v.to(torch.bfloat16) if isinstance(v, torch.Tensor) and v.dtype == torch.float32 else v)
            for k, v in d.items()}


def _tm(d, time_major):
    return {k: (synth.to_time_major(v) if time_major and isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _shift(d):
    """Copies of the [.., T, ..] tensors one element past an aligned base:
    4-byte (1-byte for flags) rather than 16-byte aligned."""
    out = {}
    for k, v in d.items():
        if isinstance(v, torch.Tensor) and v.dim() >= 2:
            buf = torch.empty(v.numel() + 16, dtype=v.dtype, device=v.device)
            view = buf[1:1 + v.numel()].view(v.shape)
            view.copy_(v)
            out[k] = view
        else:
            out[k] = v
    return out


def _back(t, time_major):
    return synth.from_time_major(t) if time_major else t


KINDS = ["gae", "disc", "td", "vt", "vtrace", "retrace", "elig", "psum_i32", "psum_f32", "affine_bwd",
         "affine_fwd"]


def make_inputs(kind, E, T, seed, trunc, device, **kw):
    if kind in ("gae", "disc", "td", "vt"):
        return synth.value_rollout(E, T, seed, p_term=kw.get("p_term", 0.01), p_trunc=kw.get("p_trunc", 0.005),
                                   with_trunc=trunc, device=device)
    if kind == "vtrace":
        return synth.vtrace_rollout(E, T, seed, p_term=kw.get("p_term", 0.01), p_trunc=0.005 if trunc else 0.0,
                                    with_trunc=trunc, device=device)
    if kind == "retrace":
        return synth.retrace_rollout(E, T, seed, p_term=kw.get("p_term", 0.002), p_trunc=0.005 if trunc else 0.0,
                                     with_trunc=trunc, num_actions=kw.get("num_actions", synth.NUM_ACTIONS),
                                     device=device)
    if kind in ("elig", "psum_i32", "psum_f32"):
        return synth.forward_rollout(E, T, seed, p_term=kw.get("p_term", 0.01), p_trunc=0.005, with_trunc=trunc,
                                     device=device)
    if kind in ("affine_bwd", "affine_fwd"):
        return synth.affine_rollout(E, T, seed, device=device)
    raise ValueError(kind)


def run_gpu(kind, d, time_major=False, multipass=False, params=None, inputs_ready=False, shift=False):
    """Outputs of the CUDA path as env-major tensors (tuple).  shift: pass
    the inputs, in the call's layout, at unaligned addresses."""
    p = dict(gamma=GAMMA, lambda_=LAMBDA)
    p.update(params or {})
    x = _tm(d, time_major)
    if shift:
        x = _shift(x)
    common = dict(time_major=time_major, multipass=multipass, inputs_ready=inputs_ready)
    if kind == "gae":
        out = rlca.rlca_gae(x["rewards"], x["values"], x["terminated"], x["truncated"], x["trunc_value"],
                            x["bootstrap"], gamma=p["gamma"], lambda_=p["lambda_"], **common)
    elif kind == "vt":
        out = rlca.rlca_value_targets(x["rewards"], x["values"], x["terminated"], x["truncated"], x["trunc_value"],
                                      x["bootstrap"], gamma=p["gamma"], lambda_=p["lambda_"], **common)
    elif kind == "disc":
        out = (rlca.rlca_discounted_return(x["rewards"], x["terminated"], x["truncated"], x["trunc_value"],
                                           x["bootstrap"], gamma=p["gamma"], **common),)
    elif kind == "td":
        out = (rlca.rlca_td_lambda(x["rewards"], x["values"], x["terminated"], x["truncated"], x["trunc_value"],
                                   x["bootstrap"], gamma=p["gamma"], lambda_=p["lambda_"], **common),)
    elif kind == "vtrace":
        out = rlca.rlca_vtrace(x["rewards"], x["values"], x["logp_target"], x["logp_behaviour"], x["terminated"],
                               x["truncated"], x["trunc_value"], x["bootstrap"], gamma=p["gamma"],
                               rho_bar=p.get("rho_bar", 1.0), c_bar=p.get("c_bar", 1.0),
                               lambda_=p.get("vt_lambda", 1.0), **common)
    elif kind == "retrace":
        out = (rlca.rlca_retrace(x["q"], x["pi"], x["mu_a"], x["actions"], x["rewards"], x["terminated"],
                                 x["truncated"], x["trunc_value"], x["bootstrap"], gamma=p["gamma"],
                                 lambda_=p["lambda_"], **common),)
    elif kind == "elig":
        out = (rlca.rlca_elig_trace(x["x_f32"], x["terminated"], x["truncated"], gamma=p["gamma"],
                                    lambda_=p["lambda_"], **common),)
    elif kind in ("psum_i32", "psum_f32"):
        xs = x["x_i32"] if kind == "psum_i32" else x["x_f32"]
        out = (rlca.rlca_episodic_prefix_sum(xs, x["terminated"], x["truncated"],
                                             exclusive=p.get("exclusive", False),
                                             flag_is_start=p.get("flag_is_start", False), **common),)
    elif kind in ("affine_bwd", "affine_fwd"):
        out = (rlca.rlca_affine_scan(x["alpha"], x["beta"], x["carry"], reverse=kind == "affine_bwd", **common),)
    else:
        raise ValueError(kind)
    return tuple(None if o is None else _back(o, time_major) for o in out)


def run_oracle(kind, d, rows, params=None):
    p = dict(gamma=GAMMA, lambda_=LAMBDA)
    p.update(params or {})
    n = {k: _np(v, rows) for k, v in d.items()}
    g, lam = p["gamma"], p["lambda_"]
    if kind == "gae":
        return ref.gae(n["rewards"], n["values"], n["terminated"], n["truncated"], n["trunc_value"], n["bootstrap"],
                       gamma=g, lam=lam)
    if kind == "vt":
        adv, ret = ref.gae(n["rewards"], n["values"], n["terminated"], n["truncated"], n["trunc_value"],
                           n["bootstrap"], gamma=g, lam=lam)
        disc = ref.discounted_return(n["rewards"], n["terminated"], n["truncated"], n["trunc_value"],
                                     n["bootstrap"], gamma=g)
        td = ref.td_lambda(n["rewards"], n["values"], n["terminated"], n["truncated"], n["trunc_value"],
                           n["bootstrap"], gamma=g, lam=lam)
        return adv, ret, disc, td
    if kind == "disc":
        return (ref.discounted_return(n["rewards"], n["terminated"], n["truncated"], n["trunc_value"],
                                      n["bootstrap"], gamma=g),)
    if kind == "td":
        return (ref.td_lambda(n["rewards"], n["values"], n["terminated"], n["truncated"], n["trunc_value"],
                              n["bootstrap"], gamma=g, lam=lam),)
    if kind == "vtrace":
        return ref.vtrace(n["rewards"], n["values"], n["logp_target"], n["logp_behaviour"], n["terminated"],
                          n["truncated"], n["trunc_value"], n["bootstrap"], gamma=g,
                          rho_bar=p.get("rho_bar", 1.0), c_bar=p.get("c_bar", 1.0), lam=p.get("vt_lambda", 1.0))
    if kind == "retrace":
        return (ref.retrace(n["q"], n["pi"], n["mu_a"], n["actions"], n["rewards"], n["terminated"], n["truncated"],
                            n["trunc_value"], n["bootstrap"], gamma=g, lam=lam),)
    if kind == "elig":
        return (ref.eligibility_trace(n["x_f32"], n["terminated"], n["truncated"], gamma=g, lam=lam),)
    if kind in ("psum_i32", "psum_f32"):
        xs = n["x_i32"] if kind == "psum_i32" else n["x_f32"]
        return (ref.episodic_prefix_sum(xs, n["terminated"], n["truncated"], exclusive=p.get("exclusive", False),
                                        flag_is_start=p.get("flag_is_start", False)),)
    if kind in ("affine_bwd", "affine_fwd"):
        return (ref.affine_scan(n["alpha"], n["beta"], n["carry"], reverse=kind == "affine_bwd"),)
    raise ValueError(kind)


def check_case(kind, E, T, seed=0, trunc=True, time_major=False, multipass=False, params=None, device="cuda",
               gen_device=None, rows=None, inputs=None, inputs_ready=False, shift=False, bf16=False, **gen_kw):
    """Run one parity case; returns the worst relative error seen.  bf16:
    inputs rounded to bfloat16 and passed as such (RLCA_BF16); outputs
    checked against the oracle on those inputs with the rounding bound."""
    d = inputs if inputs is not None else make_inputs(kind, E, T, seed, trunc, gen_device or device, **gen_kw)
    d = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    if bf16:
        d = to_bf16(d)
    got = run_gpu(kind, d, time_major=time_major, multipass=multipass, params=params, inputs_ready=inputs_ready,
                  shift=shift)
    torch.cuda.synchronize()
    if rows is None:
        rows = sample_rows(E, T, seed)
    want = run_oracle(kind, d, rows, params=params)
    worst = 0.0
    for i, (g, w) in enumerate(zip(got, want)):
        if g is None:
            continue
        if bf16 and g.dtype != torch.bfloat16 and g.is_floating_point():
            raise AssertionError(f"{kind} out{i}: dtype {g.dtype}, expected bfloat16")
        worst = max(worst, assert_close(_np(g, rows), w, f"{kind} out{i} E={E} T={T} tm={time_major} "
                                                          f"trunc={trunc} mp={multipass} bf16={bf16}",
                                        tol=BF16_TOL if bf16 else TOL, rel=BF16_REL if bf16 else 0.0))
    return worst

"""PyTorch-facing wrappers of the C ABI, one per entry point, same names.

Each wrapper checks dtypes, devices and contiguity, allocates the outputs
(unless given) and the two-pass workspace, and makes one entry-point call
into ``librlca.so`` on the current CUDA stream (plus, the first time a shape
is seen, a workspace-size query whose answer is kept).  No arithmetic of
the method runs here; a missing library raises (see
:func:`first_order_linear_gb300._lib.load`).

Layout: env-major ``[E, T]`` by default; ``time_major=True`` takes ``[T, E]``
(and ``[T, E, A]`` for Retrace's per-action tensors).  ``inputs_ready=True``
sets RLCA_INPUTS_READY (the inputs were not written by the kernel just before
this call on the stream, so the call may overlap it).  Flags may be uint8 or
bool tensors; ``None`` means "no such flag" for the optional inputs.  Float
tensors are float32, or all bfloat16 (RLCA_BF16: bfloat16 storage, float32
arithmetic, outputs rounded once).
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib
from ._lib import check

__all__ = [
    "rlca_gae", "rlca_value_targets", "rlca_discounted_return", "rlca_td_lambda", "rlca_vtrace", "rlca_retrace",
    "rlca_elig_trace", "rlca_episodic_prefix_sum", "rlca_affine_scan", "rlca_workspace_size",
]


def _require_cuda(dev):
    """The call's tensors (all on ``dev`` by the checks before) must be on a
    CUDA device: the kernels read device memory and there is no host
    implementation."""
    if dev.type != "cuda":
        raise ValueError(f"tensors are on {dev}: the kernels need tensors on a CUDA device")


def _ptr(t):
    # a plain int: the entry points' argtypes turn it into a void*
    return None if t is None else t.data_ptr()


def _check(t, name, dtypes, shape, device, required=True):
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return
    # one combined test on the common path; the detailed checks name the fault
    if (isinstance(t, torch.Tensor) and t.dtype in dtypes and t.shape == shape and t.device == device
            and t.is_contiguous()):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {dtypes}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_F = (torch.float32,)
_U8 = (torch.uint8, torch.bool)
_I32 = (torch.int32,)


def _fdt(t, name):
    """Element type of a call's float arrays, taken from its first float
    input: float32, or bfloat16 (RLCA_BF16: bfloat16 storage, float32
    arithmetic).  Every other float tensor of the call must match."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"{name}: dtype {t.dtype}, expected float32 or bfloat16")
    return t.dtype


def _fflag(fdt):
    return _lib.RLCA_BF16 if fdt == torch.bfloat16 else 0


def _flags(time_major, multipass, extra=0, inputs_ready=False):
    return ((_lib.RLCA_TIME_MAJOR if time_major else 0) | (_lib.RLCA_MULTIPASS if multipass else 0)
            | (_lib.RLCA_INPUTS_READY if inputs_ready else 0) | extra)


def _dims(x, time_major):
    if x.dim() < 2:
        raise ValueError("rollout tensors are 2-D ([E, T] or [T, E])")
    return (x.shape[1], x.shape[0]) if time_major else (x.shape[0], x.shape[1])


# workspace sizes by (estimator, E, T, A, flags, device index): a size
# depends only on these and the device's SM count, so each is asked once
_ws_sizes = {}


def rlca_workspace_size(estimator: int, E: int, T: int, num_actions: int = 0, flags: int = 0,
                        device=None) -> int:
    """Bytes of workspace a call needs on ``device`` (default: current)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    index = dev.index if dev.index is not None else torch.cuda.current_device()
    key = (estimator, E, T, num_actions, flags, index)
    need = _ws_sizes.get(key)
    if need is None:
        if len(_ws_sizes) >= 4096:  # many distinct shapes: start over rather than grow without bound
            _ws_sizes.clear()
        lib = _lib.load()
        out = C.c_size_t(0)
        with torch.cuda.device(index):
            check("rlca_workspace_size", lib.rlca_workspace_size(estimator, E, T, num_actions, flags, C.byref(out)))
        need = _ws_sizes[key] = out.value
    return need


def _workspace(estimator, E, T, A, flags, device, workspace):
    need = rlca_workspace_size(estimator, E, T, A, flags, device)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < need or workspace.device != device:
        raise ValueError(f"workspace needs {need} bytes on {device}")
    return workspace, workspace.numel() * workspace.element_size()


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _hold(device, stream, *tensors):
    """Marks device tensors the call reads or writes as in use on ``stream``
    when that is not the current stream.  Buffers this module allocates
    (the workspace, outputs not passed in) come from the caching allocator
    on the current stream; without the mark, memory freed there could be
    handed to new work on the current stream while the kernel on ``stream``
    still reads or writes it."""
    if stream is None or stream == torch.cuda.current_stream(device):
        return
    for t in tensors:
        if t is not None:
            t.record_stream(stream)


def _boundaries(shape, dev, terminated, truncated, trunc_value, bootstrap, E, F=_F):
    _check(terminated, "terminated", _U8, shape, dev, required=False)
    _check(truncated, "truncated", _U8, shape, dev, required=False)
    _check(trunc_value, "trunc_value", F, shape, dev, required=truncated is not None)
    _check(bootstrap, "bootstrap", F, (E,), dev, required=False)


def rlca_gae(rewards, values, terminated=None, truncated=None, trunc_value=None, bootstrap=None, *,
             gamma=0.99, lambda_=0.95, advantages=None, returns=None, want_returns=True,
             time_major=False, multipass=False, inputs_ready=False, workspace=None, stream=None):
    """GAE advantages (and returns = advantages + values).  Returns
    ``(advantages, returns)``; returns is None when ``want_returns`` is
    False and no buffer is given."""
    lib = _lib.load()
    dev = rewards.device
    fdt = _fdt(rewards, "rewards")
    F = (fdt,)
    E, T = _dims(rewards, time_major)
    shape = tuple(rewards.shape)
    _check(rewards, "rewards", F, shape, dev)
    _check(values, "values", F, shape, dev)
    _boundaries(shape, dev, terminated, truncated, trunc_value, bootstrap, E, F)
    if advantages is None:
        advantages = torch.empty(shape, dtype=fdt, device=dev)
    if returns is None and want_returns:
        returns = torch.empty(shape, dtype=fdt, device=dev)
    _check(advantages, "advantages", F, shape, dev)
    _check(returns, "returns", F, shape, dev, required=False)
    flags = _flags(time_major, multipass, inputs_ready=inputs_ready) | _fflag(fdt)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_GAE, E, T, 0, flags, dev, workspace)
        check("rlca_gae", lib.rlca_gae(
            _ptr(rewards), _ptr(values), _ptr(terminated), _ptr(truncated), _ptr(trunc_value), _ptr(bootstrap),
            _ptr(advantages), _ptr(returns), E, T, gamma, lambda_, flags, _ptr(ws), wsb, _stream(dev, stream)))
        _hold(dev, stream, ws, advantages, returns)
    return advantages, returns


def rlca_value_targets(rewards, values, terminated=None, truncated=None, trunc_value=None, bootstrap=None, *,
                       gamma=0.99, lambda_=0.95, advantages=None, returns=None, disc_returns=None,
                       td_lambda_returns=None, outputs=("advantages", "returns", "disc_returns", "td_lambda_returns"),
                       time_major=False, multipass=False, inputs_ready=False, workspace=None, stream=None):
    """GAE advantages and returns, discounted returns and TD(lambda) returns
    in one fused pass.  ``outputs`` names the results to compute (buffers
    passed explicitly are always written).  Returns the four tensors (None
    for those not computed) in the order (advantages, returns,
    disc_returns, td_lambda_returns)."""
    lib = _lib.load()
    dev = rewards.device
    fdt = _fdt(rewards, "rewards")
    F = (fdt,)
    E, T = _dims(rewards, time_major)
    shape = tuple(rewards.shape)
    _check(rewards, "rewards", F, shape, dev)
    _check(values, "values", F, shape, dev)
    _boundaries(shape, dev, terminated, truncated, trunc_value, bootstrap, E, F)
    bufs = dict(advantages=advantages, returns=returns, disc_returns=disc_returns,
                td_lambda_returns=td_lambda_returns)
    for name in bufs:
        if bufs[name] is None and name in outputs:
            bufs[name] = torch.empty(shape, dtype=fdt, device=dev)
        _check(bufs[name], name, F, shape, dev, required=False)
    flags = _flags(time_major, multipass, inputs_ready=inputs_ready) | _fflag(fdt)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_VALUE_TARGETS, E, T, 0, flags, dev, workspace)
        check("rlca_value_targets", lib.rlca_value_targets(
            _ptr(rewards), _ptr(values), _ptr(terminated), _ptr(truncated), _ptr(trunc_value), _ptr(bootstrap),
            _ptr(bufs["advantages"]), _ptr(bufs["returns"]), _ptr(bufs["disc_returns"]),
            _ptr(bufs["td_lambda_returns"]), E, T, gamma, lambda_, flags, _ptr(ws), wsb, _stream(dev, stream)))
        _hold(dev, stream, ws, *bufs.values())
    return bufs["advantages"], bufs["returns"], bufs["disc_returns"], bufs["td_lambda_returns"]


def rlca_discounted_return(rewards, terminated=None, truncated=None, trunc_value=None, bootstrap=None, *,
                           gamma=0.99, out=None, time_major=False, multipass=False, inputs_ready=False, workspace=None,
                           stream=None):
    """Discounted returns G_t = r_t + gamma * G_{t+1} with the boundary rules."""
    lib = _lib.load()
    dev = rewards.device
    fdt = _fdt(rewards, "rewards")
    F = (fdt,)
    E, T = _dims(rewards, time_major)
    shape = tuple(rewards.shape)
    _check(rewards, "rewards", F, shape, dev)
    _boundaries(shape, dev, terminated, truncated, trunc_value, bootstrap, E, F)
    if out is None:
        out = torch.empty(shape, dtype=fdt, device=dev)
    _check(out, "out", F, shape, dev)
    flags = _flags(time_major, multipass, inputs_ready=inputs_ready) | _fflag(fdt)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_DISCOUNTED_RETURN, E, T, 0, flags, dev, workspace)
        check("rlca_discounted_return", lib.rlca_discounted_return(
            _ptr(rewards), _ptr(terminated), _ptr(truncated), _ptr(trunc_value), _ptr(bootstrap), _ptr(out),
            E, T, gamma, flags, _ptr(ws), wsb, _stream(dev, stream)))
        _hold(dev, stream, ws, out)
    return out


def rlca_td_lambda(rewards, values, terminated=None, truncated=None, trunc_value=None, bootstrap=None, *,
                   gamma=0.99, lambda_=0.95, out=None, time_major=False, multipass=False, inputs_ready=False, workspace=None,
                   stream=None):
    """TD(lambda) returns."""
    lib = _lib.load()
    dev = rewards.device
    fdt = _fdt(rewards, "rewards")
    F = (fdt,)
    E, T = _dims(rewards, time_major)
    shape = tuple(rewards.shape)
    _check(rewards, "rewards", F, shape, dev)
    _check(values, "values", F, shape, dev)
    _boundaries(shape, dev, terminated, truncated, trunc_value, bootstrap, E, F)
    if out is None:
        out = torch.empty(shape, dtype=fdt, device=dev)
    _check(out, "out", F, shape, dev)
    flags = _flags(time_major, multipass, inputs_ready=inputs_ready) | _fflag(fdt)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_TD_LAMBDA, E, T, 0, flags, dev, workspace)
        check("rlca_td_lambda", lib.rlca_td_lambda(
            _ptr(rewards), _ptr(values), _ptr(terminated), _ptr(truncated), _ptr(trunc_value), _ptr(bootstrap),
            _ptr(out), E, T, gamma, lambda_, flags, _ptr(ws), wsb, _stream(dev, stream)))
        _hold(dev, stream, ws, out)
    return out


def rlca_vtrace(rewards, values, logp_target, logp_behaviour, terminated=None, truncated=None,
                trunc_value=None, bootstrap=None, *, gamma=0.99, rho_bar=1.0, c_bar=1.0, lambda_=1.0,
                vs=None, pg_advantages=None, want_pg=True, time_major=False, multipass=False, inputs_ready=False,
                workspace=None, stream=None):
    """V-Trace targets and policy-gradient advantages: ``(vs, pg_advantages)``."""
    lib = _lib.load()
    dev = rewards.device
    fdt = _fdt(rewards, "rewards")
    F = (fdt,)
    E, T = _dims(rewards, time_major)
    shape = tuple(rewards.shape)
    for name, t in (("rewards", rewards), ("values", values), ("logp_target", logp_target),
                    ("logp_behaviour", logp_behaviour)):
        _check(t, name, F, shape, dev)
    _boundaries(shape, dev, terminated, truncated, trunc_value, bootstrap, E, F)
    if vs is None:
        vs = torch.empty(shape, dtype=fdt, device=dev)
    if pg_advantages is None and want_pg:
        pg_advantages = torch.empty(shape, dtype=fdt, device=dev)
    _check(vs, "vs", F, shape, dev)
    _check(pg_advantages, "pg_advantages", F, shape, dev, required=False)
    flags = _flags(time_major, multipass, inputs_ready=inputs_ready) | _fflag(fdt)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_VTRACE, E, T, 0, flags, dev, workspace)
        check("rlca_vtrace", lib.rlca_vtrace(
            _ptr(rewards), _ptr(values), _ptr(logp_target), _ptr(logp_behaviour), _ptr(terminated),
            _ptr(truncated), _ptr(trunc_value), _ptr(bootstrap), _ptr(vs), _ptr(pg_advantages), E, T,
            gamma, rho_bar, c_bar, lambda_, flags, _ptr(ws), wsb, _stream(dev, stream)))
        _hold(dev, stream, ws, vs, pg_advantages)
    return vs, pg_advantages


def rlca_retrace(q, pi, mu_a, actions, rewards, terminated=None, truncated=None, trunc_value=None,
                 bootstrap=None, *, gamma=0.99, lambda_=0.95, out=None, time_major=False, multipass=False, inputs_ready=False,
                 workspace=None, stream=None):
    """Retrace(lambda) Q targets; q and pi are [E, T, A] ([T, E, A])."""
    lib = _lib.load()
    dev = rewards.device
    fdt = _fdt(rewards, "rewards")
    F = (fdt,)
    E, T = _dims(rewards, time_major)
    shape = tuple(rewards.shape)
    if q.dim() != 3:
        raise ValueError("q must be 3-D")
    A = q.shape[-1]
    _check(q, "q", F, shape + (A,), dev)
    _check(pi, "pi", F, shape + (A,), dev)
    _check(mu_a, "mu_a", F, shape, dev)
    _check(actions, "actions", _I32, shape, dev)
    _check(rewards, "rewards", F, shape, dev)
    _boundaries(shape, dev, terminated, truncated, trunc_value, bootstrap, E, F)
    if out is None:
        out = torch.empty(shape, dtype=fdt, device=dev)
    _check(out, "out", F, shape, dev)
    flags = _flags(time_major, multipass, inputs_ready=inputs_ready) | _fflag(fdt)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_RETRACE, E, T, A, flags, dev, workspace)
        check("rlca_retrace", lib.rlca_retrace(
            _ptr(q), _ptr(pi), _ptr(mu_a), _ptr(actions), _ptr(rewards), _ptr(terminated), _ptr(truncated),
            _ptr(trunc_value), _ptr(bootstrap), _ptr(out), E, T, A, gamma, lambda_, flags, _ptr(ws), wsb,
            _stream(dev, stream)))
        _hold(dev, stream, ws, out)
    return out


def rlca_elig_trace(x, terminated=None, truncated=None, *, gamma=0.99, lambda_=0.95, out=None,
                    time_major=False, multipass=False, inputs_ready=False, workspace=None, stream=None):
    """Accumulating eligibility trace (forward scan)."""
    lib = _lib.load()
    dev = x.device
    fdt = _fdt(x, "x")
    F = (fdt,)
    E, T = _dims(x, time_major)
    shape = tuple(x.shape)
    _check(x, "x", F, shape, dev)
    _check(terminated, "terminated", _U8, shape, dev, required=False)
    _check(truncated, "truncated", _U8, shape, dev, required=False)
    if out is None:
        out = torch.empty(shape, dtype=fdt, device=dev)
    _check(out, "out", F, shape, dev)
    flags = _flags(time_major, multipass, inputs_ready=inputs_ready) | _fflag(fdt)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_ELIG_TRACE, E, T, 0, flags, dev, workspace)
        check("rlca_elig_trace", lib.rlca_elig_trace(
            _ptr(x), _ptr(terminated), _ptr(truncated), _ptr(out), E, T, gamma, lambda_, flags, _ptr(ws), wsb,
            _stream(dev, stream)))
        _hold(dev, stream, ws, out)
    return out


def rlca_episodic_prefix_sum(x, terminated=None, truncated=None, *, exclusive=False, flag_is_start=False,
                             out=None, time_major=False, multipass=False, inputs_ready=False, workspace=None, stream=None):
    """Per-episode running sum of x (int32 wraps; float32 or bfloat16 storage)."""
    lib = _lib.load()
    dev = x.device
    E, T = _dims(x, time_major)
    shape = tuple(x.shape)
    if x.dtype == torch.int32:
        dtype = _lib.RLCA_I32
    elif x.dtype in (torch.float32, torch.bfloat16):
        dtype = _lib.RLCA_F32
    else:
        raise TypeError("x must be int32, float32 or bfloat16")
    _check(x, "x", (x.dtype,), shape, dev)
    _check(terminated, "terminated", _U8, shape, dev, required=False)
    _check(truncated, "truncated", _U8, shape, dev, required=False)
    if out is None:
        out = torch.empty(shape, dtype=x.dtype, device=dev)
    _check(out, "out", (x.dtype,), shape, dev)
    extra = (_lib.RLCA_PSUM_EXCLUSIVE if exclusive else 0) | (_lib.RLCA_PSUM_FLAG_IS_START if flag_is_start else 0)
    flags = _flags(time_major, multipass, extra, inputs_ready=inputs_ready) | (
        _lib.RLCA_BF16 if x.dtype == torch.bfloat16 else 0)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_PREFIX_SUM, E, T, 0, flags, dev, workspace)
        check("rlca_episodic_prefix_sum", lib.rlca_episodic_prefix_sum(
            _ptr(x), dtype, _ptr(terminated), _ptr(truncated), _ptr(out), E, T, flags, _ptr(ws), wsb,
            _stream(dev, stream)))
        _hold(dev, stream, ws, out)
    return out


def rlca_affine_scan(alpha, beta, carry=None, *, reverse=True, out=None, time_major=False, multipass=False, inputs_ready=False,
                     workspace=None, stream=None):
    """Generic A_t = alpha_t + beta_t * A_{t+1} (reverse) or A_{t-1} (forward)."""
    lib = _lib.load()
    dev = alpha.device
    fdt = _fdt(alpha, "alpha")
    F = (fdt,)
    E, T = _dims(alpha, time_major)
    shape = tuple(alpha.shape)
    _check(alpha, "alpha", F, shape, dev)
    _check(beta, "beta", F, shape, dev)
    _check(carry, "carry", F, (E,), dev, required=False)
    if out is None:
        out = torch.empty(shape, dtype=fdt, device=dev)
    _check(out, "out", F, shape, dev)
    flags = _flags(time_major, multipass, inputs_ready=inputs_ready) | _fflag(fdt)
    _require_cuda(dev)
    with torch.cuda.device(dev):
        ws, wsb = _workspace(_lib.RLCA_EST_AFFINE_SCAN, E, T, 0, flags, dev, workspace)
        check("rlca_affine_scan", lib.rlca_affine_scan(
            _ptr(alpha), _ptr(beta), _ptr(carry), _ptr(out), E, T, 1 if reverse else 0, flags, _ptr(ws), wsb,
            _stream(dev, stream)))
        _hold(dev, stream, ws, out)
    return out

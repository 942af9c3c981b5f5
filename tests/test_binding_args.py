"""Argument checks of the Python binding, on the CPU: every malformed call
raises before anything is launched, and well-formed tensors that are not on
a CUDA device raise too (there is no CPU fallback)."""
import pytest
import torch

from first_order_linear_gb300 import build, rlca

E, T, A = 4, 8, 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _f(*shape, dtype=torch.float32):
    return torch.zeros(*shape, dtype=dtype)


def _u8(*shape):
    return torch.zeros(*shape, dtype=torch.uint8)


def test_float_dtypes():
    with pytest.raises(TypeError):
        rlca.rlca_gae(_f(E, T, dtype=torch.float64), _f(E, T))
    with pytest.raises(TypeError):  # one call, one float storage type
        rlca.rlca_gae(_f(E, T), _f(E, T, dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        rlca.rlca_episodic_prefix_sum(_f(E, T, dtype=torch.float64))
    with pytest.raises(TypeError):
        rlca.rlca_episodic_prefix_sum(torch.zeros(E, T, dtype=torch.int64))
    with pytest.raises(TypeError):  # flags are uint8 or bool
        rlca.rlca_discounted_return(_f(E, T), torch.zeros(E, T, dtype=torch.int32))
    with pytest.raises(TypeError):  # actions are int32
        rlca.rlca_retrace(_f(E, T, A), _f(E, T, A), _f(E, T), torch.zeros(E, T, dtype=torch.int64), _f(E, T))


def test_shapes():
    with pytest.raises(ValueError):
        rlca.rlca_gae(_f(E, T), _f(E, T + 1))
    with pytest.raises(ValueError):
        rlca.rlca_gae(_f(T * E), _f(T * E))  # rollouts are 2-D
    with pytest.raises(ValueError):
        rlca.rlca_gae(_f(E, T), _f(E, T), bootstrap=_f(T))  # bootstrap is [E]
    with pytest.raises(ValueError):
        rlca.rlca_gae(_f(E, T), _f(E, T), time_major=True, bootstrap=_f(E))  # [T, E] input: bootstrap [T]
    with pytest.raises(ValueError):
        rlca.rlca_retrace(_f(E, T), _f(E, T), _f(E, T), torch.zeros(E, T, dtype=torch.int32), _f(E, T))
    with pytest.raises(ValueError):
        rlca.rlca_retrace(_f(E, T, A), _f(E, T, A + 1), _f(E, T), torch.zeros(E, T, dtype=torch.int32), _f(E, T))
    with pytest.raises(ValueError):
        rlca.rlca_value_targets(_f(E, T), _f(E, T), advantages=_f(E, T - 1))


def test_truncation_needs_values():
    with pytest.raises(ValueError):
        rlca.rlca_gae(_f(E, T), _f(E, T), _u8(E, T), _u8(E, T))
    with pytest.raises(ValueError):
        rlca.rlca_vtrace(_f(E, T), _f(E, T), _f(E, T), _f(E, T), None, _u8(E, T))


def test_contiguity():
    r = _f(T, E).t()  # [E, T] view, not contiguous
    with pytest.raises(ValueError):
        rlca.rlca_discounted_return(r)
    with pytest.raises(ValueError):
        rlca.rlca_elig_trace(_f(E, T), _u8(T, E).t())


def test_no_cpu_fallback():
    """Well-formed CPU tensors: the binding refuses them rather than
    computing anything on the host."""
    r, v = torch.randn(E, T), torch.randn(E, T)
    out = torch.full((E, T), 7.0)
    with pytest.raises(ValueError, match="CUDA device"):
        rlca.rlca_discounted_return(r, out=out)
    assert torch.all(out == 7.0)
    with pytest.raises(ValueError, match="CUDA device"):
        rlca.rlca_gae(r, v)
    with pytest.raises(ValueError, match="CUDA device"):
        rlca.rlca_episodic_prefix_sum(torch.zeros(E, T, dtype=torch.int32))

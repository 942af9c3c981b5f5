"""GB300-native (sm_103a) affine-scan kernels for RL credit assignment.

The seven estimators of rl-triton (arXiv:2608.17641) -- GAE, V-Trace,
Retrace(lambda), TD(lambda) returns, discounted returns, eligibility traces
and episodic prefix sums -- plus the generic affine scan, as hand-written
CUDA kernels behind the C ABI of ``include/rlca.h``.  :mod:`.rlca` holds the
PyTorch-facing wrappers (same names as the C entry points), :mod:`._lib` the
ctypes view of the library, :mod:`.build` the in-tree build, :mod:`.synth`
the seeded synthetic rollouts.
"""
from .rlca import (  # noqa: F401
    rlca_affine_scan, rlca_discounted_return, rlca_elig_trace, rlca_episodic_prefix_sum, rlca_gae,
    rlca_retrace, rlca_td_lambda, rlca_value_targets, rlca_vtrace, rlca_workspace_size,
)

__version__ = "0.1.0"

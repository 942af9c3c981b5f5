"""Float64 CPU oracle for the credit-assignment scans -- TEST INFRASTRUCTURE.

This package is the slow, obviously correct reference that the CUDA path is
checked against.  Only the test suite, the smoke check in the repository's
entry module and the CPU-baseline leg of the benchmark may import it; the
library itself never does, and it shares no code with the CUDA path.

Every function is a plain sequential loop over time steps in float64,
vectorised only across independent environments, written from the
definitions cited in its docstring.  See :mod:`oracle.rlca_ref`.
"""
from . import rlca_ref  # noqa: F401

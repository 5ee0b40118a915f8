"""Oracle for the compressed sparse attention path (test infrastructure only).

A plain fp64 numpy restatement of what the path computes.  Only the tests,
the package smoke check and the benchmark's CPU-baseline leg import it; the
library never does, and the two share no code.
"""

from . import csa_oracle  # noqa: F401
from .workload_oracle import SequenceOracle  # noqa: F401

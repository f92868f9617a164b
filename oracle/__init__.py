"""CPU oracle for the CSA2 step: test infrastructure only.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline / reference leg
of `bench.py` may import this package. The CUDA product path never does.
"""
from . import formats  # noqa: F401
from . import csa2_oracle  # noqa: F401

"""CSA2 compressed sparse attention for one GB300 (sm_103a) GPU.

The computation lives in a C-ABI CUDA library (include/csa2.h, built from
csrc/ by build.build()); `binding` is its thin Python marshalling layer.
"""
from . import build  # noqa: F401

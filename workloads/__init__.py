"""Seeded synthetic inputs for the CSA2 step.

This package only draws random numbers into the shapes, dtypes and layouts
the step consumes. It holds none of the method's arithmetic (no pooling,
scoring, selection, softmax, rotation or quantisation), so both the CUDA path
and the CPU oracle can take their inputs from it.
"""
from .gen import Workload, PRESETS, make_inputs, make_topk_scores, make_selection  # noqa: F401

"""Seeded synthetic MoE-layer workloads shared by the tests and the benchmark.

This module draws random inputs and runs the model's forward pieces that sit
OUTSIDE the recalibrated backward path (the router and the SwiGLU expert
forward that produce the saved state). It holds none of the path's steps:
no dispatch permutation, no LRM score, no selection, no compaction and no
backward. Both the CUDA path and the CPU oracle receive the same bytes it
produces.
"""

from .configs import LayerConfig, CONFIGS, get_config, with_tokens  # noqa: F401
from .generate import generate  # noqa: F401

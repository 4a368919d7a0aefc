"""Seeded synthetic inputs for the fused EXL3 routed-expert MoE layer.

This package generates random inputs only (trellis words, sign vectors, scales,
activations, router ids and weights).  It holds none of the layer's arithmetic
and is shared by the float64 oracle's tests and by the CUDA path's tests and
benchmark, so that both sides see bit-identical inputs.
"""

from .synth import *  # noqa: F401,F403

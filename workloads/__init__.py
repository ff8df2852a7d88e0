"""Seeded synthetic inputs for the MoE layer forward.

This package holds the layer shapes and the seeded tensor generators that both
the CUDA path's tests/benchmark and the float64 oracle consume.  It contains
none of the layer's arithmetic (no routing, no expert FFN): only shapes,
distributions and seeds.
"""

from .shapes import SHAPES, MoEShape, shape_by_name
from .generate import make_inputs, tensor_seed, ExpertWeights

__all__ = ["SHAPES", "MoEShape", "shape_by_name", "make_inputs", "tensor_seed",
           "ExpertWeights"]

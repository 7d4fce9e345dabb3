"""Nested-bit quantized linear layer (2-bit Lloyd-Max base + b-bit residual) for GB300.

The compute runs in ``libnest`` (hand-written sm_103a CUDA behind a C ABI,
``include/nest.h``); :mod:`nested_bit_quantized_gb300.nest` is its thin
Python binding and :mod:`nested_bit_quantized_gb300.synth` holds the seeded
synthetic inputs.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "nest", "build"]

"""Seeded synthetic inputs for the OSCAR INT2 paged-KV decode path.

This package holds input generators only: random K/V/q rows with channel
outliers, synthetic rotation bases U, sequence lengths. It contains none of the
method's arithmetic (no rotation, quantisation or attention). Both the CPU
oracle's tests and the CUDA path's tests/benchmark draw their inputs from here.
"""
from .synth import *  # noqa: F401,F403

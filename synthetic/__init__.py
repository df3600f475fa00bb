"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA-side tests.

This package holds no arithmetic of the method: it only draws random numbers
with numpy's PCG64 generator and stores bf16 values as raw uint16 bit patterns
(the fp32 -> bf16 conversion is done by torch on the CPU, round to nearest even).
"""
from .inputs import *  # noqa: F401,F403

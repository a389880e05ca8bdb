"""Seeded synthetic inputs shared by the oracle tests, the CUDA-path tests and the bench.

This package only draws random numbers and lays them out as bf16 bit patterns
(uint16 arrays).  It holds none of the layer's arithmetic: no selection, no
norms, no products.
"""
from .inputs import *  # noqa: F401,F403

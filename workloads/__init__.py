"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This package draws numbers and builds input structures (context lengths, shuffled
page assignments, request lists).  It holds none of the method's arithmetic.
"""
from . import configs, rng  # noqa: F401

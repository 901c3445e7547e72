"""Seeded synthetic inputs shared by the tests, the oracle runs and the bench.

This package draws random tensors only: it holds none of the projection's
arithmetic, and it imports neither the oracle nor the CUDA library.
"""
from .gen import *  # noqa: F401,F403

"""Seeded synthetic inputs shared by the oracle checks, the GPU tests and the
benchmark. This package draws random numbers and nothing else: it holds none
of the method's arithmetic (no decode, no transform, no matvec)."""
from .gen import *  # noqa: F401,F403

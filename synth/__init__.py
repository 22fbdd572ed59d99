"""Seeded synthetic inputs shared by the oracle tests, the CUDA tests and the benchmark."""
from . import generate  # noqa: F401

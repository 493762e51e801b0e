"""Seeded synthetic inputs shared by the oracle tests and the GPU tests.

Holds none of the method's arithmetic: only random matrices."""
from . import generators  # noqa: F401

"""Seeded synthetic inputs for the Engram hot path (shared by tests and bench; no method arithmetic)."""
from . import generators, workloads  # noqa: F401

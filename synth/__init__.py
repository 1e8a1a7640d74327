"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the benchmark.

Holds no arithmetic of the verification method: only random logits and uniforms.
"""
from . import philox, workloads  # noqa: F401

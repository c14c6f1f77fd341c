"""Seeded synthetic inputs shared by the oracle side and the GPU side of the
tests and the benchmark.  Holds no arithmetic of the cache itself."""

from .gen import InputSpec, bf16_bits, round_to_bf16  # noqa: F401

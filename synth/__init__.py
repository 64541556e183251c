"""Seeded synthetic inputs shared by the CUDA path's tests/benchmarks and the oracle.

This package draws random values and routing tables and nothing else: it holds none of
the collective's arithmetic (no summation, no rounding of sums, no layout naming).
"""

from .inputs import (  # noqa: F401
    bf16_bits_from_f32_trunc,
    uniform_bf16,
    normal_bf16,
    uniform_f32,
    normal_f32,
    small_int_bf16,
    small_int_f32,
    random_bytes,
    zipf_topk_routing,
    random_naming,
    seeded_rng,
    device_uniform_bf16,
    device_normal_bf16,
)

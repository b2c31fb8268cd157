"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This package draws random numbers and lays them out; it holds none of the
attention method's arithmetic (no pooling, no softmax, no selection).
"""
from .gen import (  # noqa: F401
    CONFIGS,
    WorkloadConfig,
    bf16_round_bits,
    bf16_bits_to_f32,
    make_head,
    make_inputs,
    token_coords,
)

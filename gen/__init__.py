"""Seeded synthetic input generators (no tail arithmetic)."""
from .workloads import Workload, custom, make, NAMED, f32_to_bf16_bits, bf16_bits_to_f32, pad_lanes  # noqa: F401

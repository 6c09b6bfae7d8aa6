"""Seeded synthetic workloads shared by the oracle tests, the GPU tests and the benchmark."""
from .synth import (Workload, WORKLOADS, make, make_segments, make_far_keys, keep_floor,
                    f32_to_bf16_bits, bf16_bits_to_f32, f32_to_e4m3_bits, to_e4m3, first_images)

__all__ = ["Workload", "WORKLOADS", "make", "make_segments", "make_far_keys", "keep_floor",
           "f32_to_bf16_bits", "bf16_bits_to_f32", "f32_to_e4m3_bits", "to_e4m3",
           "first_images"]

"""Seeded synthetic inputs shared by the CPU oracle tests, the GPU parity tests and the benchmark.

This package draws random numbers and shapes them like the workloads on the pages
(heavy-tailed K/V with planted outlier channels, RMS-normalised rows, bf16 rounding of
model activations). It holds none of the quantisation or attention arithmetic: neither
`oracle/` nor the CUDA library imports it, and it imports neither of them.
"""
from .workloads import (  # noqa: F401
    Workload, WORKLOADS, make_inputs, make_paged_inputs, ragged_lengths, bf16_bits_from_f32, f32_from_bf16_bits,
    f16_bits_from_f32, f32_from_f16_bits,
)

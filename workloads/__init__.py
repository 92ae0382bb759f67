"""Seeded synthetic inputs for the routed-expert MLP.

This package only draws random numbers and rounds them to the storage types
the library consumes (bf16 bit patterns, fp32).  It holds none of the
method's arithmetic: both the CUDA path and the CPU oracle receive the arrays
it produces, and neither imports the other.
"""
from .synth import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits_to_f64,
    f32_to_bf16_bits,
    make_inputs,
    make_inputs_fp32,
    scaled,
    zipf_group_sizes,
)

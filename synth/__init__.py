"""Seeded synthetic inputs for the SpecPrefill scoring path.

This package only draws inputs (query/key tensors as bf16 bit patterns,
prompt offsets, planted needles) and describes the workloads. It holds none
of the method's arithmetic: no attention, pooling, chunking or selection.
Both the float64 oracle and the CUDA path consume what it produces.
"""

from .workloads import WORKLOADS, Workload, get_workload
from .inputs import Inputs, make_inputs, bf16_bits_from_f32, f32_from_bf16_bits

__all__ = [
    "WORKLOADS",
    "Workload",
    "get_workload",
    "Inputs",
    "make_inputs",
    "bf16_bits_from_f32",
    "f32_from_bf16_bits",
]

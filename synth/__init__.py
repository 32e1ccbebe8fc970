"""Seeded synthetic inputs for the SpecPrefill scoring path.

This package only draws inputs (query/key tensors as bf16 bit patterns,
prompt offsets, planted needles, and the projected, normalised and rotated
keys and queries of a random-weight draft model with its block-paged cache)
and describes the workloads. It holds none of the method's arithmetic: no
attention, pooling, chunking or selection. Both the float64 oracle and the
CUDA path consume what it produces.
"""

from .workloads import WORKLOADS, Workload, get_workload
from .inputs import Inputs, make_inputs, bf16_bits_from_f32, f32_from_bf16_bits
from .draft import DRAFT_08B, DRAFT_2B, DraftShape, attention_inputs as draft_attention_inputs, page_keys

__all__ = [
    "WORKLOADS",
    "Workload",
    "get_workload",
    "Inputs",
    "make_inputs",
    "bf16_bits_from_f32",
    "f32_from_bf16_bits",
    "DraftShape",
    "DRAFT_08B",
    "DRAFT_2B",
    "draft_attention_inputs",
    "page_keys",
]

"""Seeded synthetic inputs for one decode step of grouped-query attention.

This package holds the workload shapes and the seeded random tensors that fill
them, nothing else: no RoPE, no attention, no rounding rule of the method.
Both sides draw their inputs here -- the CUDA path (tests, bench) and the fp64
oracle -- and neither imports the other.
"""

from .workloads import WORKLOADS, Workload, workload
from .generate import (
    ContiguousCase,
    PagedCase,
    TinySequence,
    U8Cache,
    make_contiguous_case,
    make_e5m2_cache,
    make_u8_cache,
    make_paged_case,
    make_tiny_sequence,
    normal,
    paged_lengths,
)

__all__ = [
    "WORKLOADS",
    "Workload",
    "workload",
    "ContiguousCase",
    "PagedCase",
    "TinySequence",
    "U8Cache",
    "make_contiguous_case",
    "make_e5m2_cache",
    "make_u8_cache",
    "make_paged_case",
    "make_tiny_sequence",
    "normal",
    "paged_lengths",
]

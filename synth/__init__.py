"""Seeded synthetic score rows shaped like the decode-step indexer workloads.

This package only draws inputs (scores, lengths, page tables). It contains none
of the top-k method's arithmetic, so both the CPU oracle and the CUDA path can
consume its output without sharing any selection code.
"""

from .workloads import (  # noqa: F401
    CONFIGS,
    PAD_VALUE,
    Workload,
    make_workload,
    make_rows,
    config_seed,
    to_bf16_bits,
    bf16_bits_to_float,
)

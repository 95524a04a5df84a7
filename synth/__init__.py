"""Seeded synthetic inputs for SnapKV prefill compression.

This package only draws inputs (queries of the observation window, keys and
values with planted "hot" spans).  It holds none of the method's arithmetic:
no scores, no pooling, no selection.  Both the CUDA path's tests/benchmark and
the CPU oracle consume the same arrays from here.
"""
from .workloads import (  # noqa: F401
    CONFIGS,
    Layer,
    bf16_round,
    bf16_to_f32,
    config_seqlens,
    make_inputs,
    make_layer,
)

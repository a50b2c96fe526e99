"""Seeded synthetic inputs for GraniKV decode-step attention.

This package only draws random numbers and lays them out (shapes, lengths, slot orders,
append schedules).  It holds none of the attention arithmetic, so both the CPU oracle's
tests and the CUDA path can take their inputs from it without sharing any of the method.
"""

from .synth import (  # noqa: F401
    Workload,
    WorkloadSpec,
    bf16_bits,
    round_to_bf16,
    make_workload,
    tiny_fp32,
    llama8b_single_prefix_16k,
    hetero_multi_prefix_k8,
    qwen_tp1_16k,
    dispatch_sweep_cell,
    small_mixed,
    medium_shared,
    NAMED,
)

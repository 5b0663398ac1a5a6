"""Seeded input generators shared by the CPU oracle and the CUDA path (inputs only)."""

from .workloads import (  # noqa: F401
    CONFIGS,
    E4M3_SPLITK_LAYERS,
    HEAD_DIM,
    Workload,
    chunked_prefill,
    e4m3_splitk_layer,
    f32_to_bf16_bits,
    f32_to_f16_bits,
    bulk_tail_decode,
    cancelling_pairs,
    long_context_decode,
    mixed_catchup_decode,
    page1_shape,
    small_paged,
    small_random,
    tiny,
)

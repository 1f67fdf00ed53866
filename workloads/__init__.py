"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

Nothing here computes attention, paging or allocation: the modules only draw
values and lengths and describe the scheduling trace.
"""

from .configs import (SEED_BASE, DecodeWorkload, Iteration, SharedPrefixWorkload,
                      TraceConfig, Work, config1, config2, config3, config3_lengths,
                      config4, lognormal_lengths, make_decode_workload,
                      make_shared_prefix_workload, pool_blocks, trace_iterations)
from .rng import BF16_NAN, f32_to_bf16_bits, generator, normal_bf16, normal_bf16_from

__all__ = [
    "SEED_BASE", "DecodeWorkload", "Iteration", "SharedPrefixWorkload", "TraceConfig",
    "Work", "config1", "config2", "config3", "config3_lengths", "config4",
    "lognormal_lengths", "make_decode_workload", "make_shared_prefix_workload", "pool_blocks",
    "trace_iterations",
    "BF16_NAN", "f32_to_bf16_bits", "generator", "normal_bf16", "normal_bf16_from",
]

"""Seeded synthetic inputs shaped like the S³R pages' rollout workloads.

This package is the only code shared by the CUDA path's tests/bench and the
CPU oracle's tests: it draws random numbers and lays them out (paged KV pool,
block tables, queries, logits, drafted tokens).  It holds none of the method's
arithmetic.
"""

from .configs import (ATTN_CONFIGS, ATTN_QWEN3_1P7B_256SEQ, ATTN_QWEN3_1P7B_28LAYER, ATTN_QWEN3_8B_128SEQ,
                      ATTN_TINY, ROLLOUT_ACCEPTANCE_MATCHED_SIGMAS, SAMPLER_CONFIGS, SAMPLER_ROLLOUT_2048SEQ,
                      SAMPLER_ROUND_256SEQ, SAMPLER_TINY, AttnConfig, SamplerConfig)
from .attention_inputs import PagedKV, make_paged_kv, make_queries, bf16_to_bits
from .sampler_inputs import SpecInputs, make_spec_inputs
from .scheduler_inputs import RolloutRequests, make_rollout_requests

__all__ = [
    "ATTN_CONFIGS",
    "SAMPLER_CONFIGS",
    "ATTN_TINY",
    "ATTN_QWEN3_1P7B_256SEQ",
    "ATTN_QWEN3_8B_128SEQ",
    "ATTN_QWEN3_1P7B_28LAYER",
    "SAMPLER_TINY",
    "SAMPLER_ROUND_256SEQ",
    "SAMPLER_ROLLOUT_2048SEQ",
    "ROLLOUT_ACCEPTANCE_MATCHED_SIGMAS",
    "AttnConfig",
    "SamplerConfig",
    "PagedKV",
    "make_paged_kv",
    "make_queries",
    "bf16_to_bits",
    "SpecInputs",
    "make_spec_inputs",
    "RolloutRequests",
    "make_rollout_requests",
]

"""Seeded synthetic inputs shaped like the S³R pages' rollout workloads.

This package is the only code shared by the CUDA path's tests/bench and the
CPU oracle's tests: it draws random numbers and lays them out (paged KV pool,
block tables, queries, logits, drafted tokens).  It holds none of the method's
arithmetic.
"""

from .configs import ATTN_CONFIGS, SAMPLER_CONFIGS, AttnConfig, SamplerConfig
from .attention_inputs import PagedKV, make_paged_kv, make_queries, bf16_to_bits
from .sampler_inputs import SpecInputs, make_spec_inputs
from .scheduler_inputs import RolloutRequests, make_rollout_requests

__all__ = [
    "ATTN_CONFIGS",
    "SAMPLER_CONFIGS",
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

"""The workloads, each named by what it is and its sizes.

Shapes follow the S³R pages' rollout setting: Qwen3-1.7B / Qwen3-8B attention
geometry, 16K / 24K maximum responses, 256 prompts x 8 responses, the 151936
token vocabulary and the sparse budget ratio 0.05 ([wispaper] "Throughput gains
with comparable task performance"), the budget sweep 0.05 .. 0.50 ([rebas]
"为什么值得关注").  The data are synthetic: no model weights or datasets.
"""

from dataclasses import dataclass
from typing import Optional, Tuple


@dataclass(frozen=True)
class AttnConfig:
    name: str
    num_seqs: int
    hist_min: int            # history length L ~ U{hist_min .. hist_max}
    hist_max: int
    q_heads: int
    kv_heads: int
    k: int                   # draft length = verify rows T
    budgets: Tuple[float, ...]
    seed: int
    head_dim: int = 128
    layers: int = 1
    capacity_tokens: Optional[int] = None   # pool pages per sequence cover this many tokens
    heavy_per_head: int = 8
    heavy_score: float = 4.0


@dataclass(frozen=True)
class SamplerConfig:
    name: str
    num_seqs: int
    k: int
    vocab: int
    p_sigma: float
    q_sigmas: Tuple[float, ...]
    seed: int
    philox_seed: int = 0


# Attention workloads.
ATTN_TINY = AttnConfig("tiny-1layer-4x2048", num_seqs=4, hist_min=2048, hist_max=2048,
                       q_heads=16, kv_heads=8, k=4, budgets=(0.10,), seed=1)
ATTN_QWEN3_1P7B_256SEQ = AttnConfig("qwen3-1.7b-geom-256seq-4k16k", num_seqs=256, hist_min=4096, hist_max=16384,
                                    q_heads=16, kv_heads=8, k=4, budgets=(0.05,), seed=2)
ATTN_QWEN3_8B_128SEQ = AttnConfig("qwen3-8b-geom-128seq-8k24k", num_seqs=128, hist_min=8192, hist_max=24576,
                                  q_heads=32, kv_heads=8, k=8, budgets=(0.05, 0.10, 0.25, 0.50), seed=3)
ATTN_QWEN3_1P7B_28LAYER = AttnConfig("qwen3-1.7b-geom-28layer-32seq-4k16k", num_seqs=32, hist_min=4096,
                                     hist_max=16384, q_heads=16, kv_heads=8, k=4, budgets=(0.05,), seed=5,
                                     layers=28, capacity_tokens=16384)

# Sampler workloads.
SAMPLER_TINY = SamplerConfig("tiny-4seq-k4-v4096", num_seqs=4, k=4, vocab=4096, p_sigma=3.0,
                             q_sigmas=(0.5,), seed=1)
# The sampler leg of the one-layer round (sequences of the 1.7B-geometry
# workload, k = 4, Qwen3 vocabulary, sigma = 1.0).
SAMPLER_ROUND_256SEQ = SamplerConfig("round-256seq-k4-v151936", num_seqs=256, k=4, vocab=151936, p_sigma=3.0,
                                     q_sigmas=(1.0,), seed=2)
SAMPLER_ROLLOUT_2048SEQ = SamplerConfig("rollout-2048seq-k8-v151936", num_seqs=2048, k=8, vocab=151936,
                                        p_sigma=3.0, q_sigmas=(0.3, 1.0), seed=4)
# Draft-noise levels at which this recipe gives the ~95% and ~80% per-position
# acceptance the rollout workload aims for (sum_v min(p, q) = 0.951 and 0.806
# over V = 151936, p ~ N(0, 3^2)); the recipe's own 0.3 and 1.0 give 0.88 and 0.62.
ROLLOUT_ACCEPTANCE_MATCHED_SIGMAS = (0.12, 0.5)

ATTN_CONFIGS = {c.name: c for c in (ATTN_TINY, ATTN_QWEN3_1P7B_256SEQ, ATTN_QWEN3_8B_128SEQ, ATTN_QWEN3_1P7B_28LAYER)}
SAMPLER_CONFIGS = {c.name: c for c in (SAMPLER_TINY, SAMPLER_ROUND_256SEQ, SAMPLER_ROLLOUT_2048SEQ)}

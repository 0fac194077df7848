"""Synthetic RL rollout requests for the scheduler simulation.

Recipe: n_prompts prompts of
U{prompt_lo .. prompt_hi} tokens, each sampled `group` times (a response
group shares its prompt); response lengths log-uniform on
[response_lo, response_hi] (long-tailed, as in long-context reasoning);
each S³R round of a request emits n_acc + 1 tokens, where n_acc counts the
leading accepted drafts among k independent acceptances of probability
`alpha` (per-position acceptance).  Enough rounds are drawn to cover the
response.  All randomness from one numpy Generator, seeded.
"""

from dataclasses import dataclass

import numpy as np


@dataclass
class RolloutRequests:
    prompt_lens: np.ndarray     # [R] int32
    response_lens: np.ndarray   # [R] int32
    emits: list                 # R arrays of int32, tokens emitted per round

    @property
    def n(self):
        return len(self.prompt_lens)


def make_rollout_requests(n_prompts, group, seed, prompt_lo=512, prompt_hi=2048, response_lo=512,
                          response_hi=16384, k=4, alpha=0.8):
    rng = np.random.default_rng(seed)
    R = n_prompts * group
    prompts = np.repeat(rng.integers(prompt_lo, prompt_hi + 1, size=n_prompts), group).astype(np.int32)
    responses = np.exp(rng.uniform(np.log(response_lo), np.log(response_hi), size=R)).astype(np.int32)
    responses = np.maximum(responses, 1)
    emits = []
    for r in range(R):
        out, total = [], 0
        while total < responses[r]:
            n = max(16, int((responses[r] - total) / 2) + 8)
            ok = rng.random((n, k)) < alpha
            e = np.cumprod(ok, axis=1).sum(axis=1) + 1
            out.append(e.astype(np.int32))
            total += int(e.sum())
        emits.append(np.concatenate(out))
    return RolloutRequests(prompts, responses.astype(np.int32), emits)

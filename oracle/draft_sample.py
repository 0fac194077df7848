"""Oracle for sampling a draft token from the drafter's logits.

Test infrastructure only (see the package docstring).

The drafter proposes each token by sampling from its own (sparse-attention)
distribution q ([wispaper] "S3R drafts sparsely and verifies densely": the
drafter proposes several tokens; [rebas] "草稿可以稀疏，交卷必须完整").  Draft
step j of sequence n draws its token from q = softmax(logits) at temperature
1, by the inverse CDF in token-id order at the Philox uniform of counter
(n, j, DRAFT, offset) — the same conventions as the verification sampler
(spec_sample.py), on the DRAFT stream.

  token = the smallest v with C_v > u * C_last, C the inclusive prefix sums
          of q in token-id order.

Parity status: pinned by tests/test_oracle_draft_sample.py: uniform logits
give token = floor(u * V) exactly; a dominant logit is always drawn; the
drawn tokens follow softmax(logits) (chi-square over 10^6 sequences).
"""

import numpy as np

from .philox import philox_uniform, STREAM_DRAFT


def sample_draft_tokens(logits, seed, offset, draft_pos, seq_ids=None):
    """logits [N][V] (or [1][V] broadcast to seq_ids) -> tokens [N] int64 and
    a dict with the uniforms and the row totals used by tests for ties."""
    x = np.asarray(logits, dtype=np.float64)
    n_rows, V = x.shape
    ids = np.arange(n_rows) if seq_ids is None else np.asarray(seq_ids, dtype=np.int64)
    N = len(ids)
    rows = np.arange(N) if n_rows == N else np.zeros(N, dtype=np.int64)
    m = x.max(axis=1, keepdims=True)
    e = np.exp(x - m)
    q = e / e.sum(axis=1, keepdims=True)
    cdf = np.cumsum(q[rows], axis=1)
    total = cdf[:, -1]
    u = philox_uniform(seed, offset, ids, int(draft_pos), STREAM_DRAFT)
    target = u * total
    tokens = np.argmax(cdf > target[:, None], axis=1)
    return tokens.astype(np.int64), {"u": u, "total": total, "target": target, "cdf_rows": rows}

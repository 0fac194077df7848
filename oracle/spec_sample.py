"""Oracle for exact speculative sampling of one drafted block.

Test infrastructure only (see the package docstring).

The pages fix the method: the target policy verifies the drafted tokens through
exact speculative sampling, which keeps the output distributed as the dense
policy ([wispaper] "S3R drafts sparsely and verifies densely"); a draft that
fails is replaced by a token resampled from the corrected distribution
([rebas] "草稿可以稀疏，交卷必须完整"); after the first rejection the correcting
token comes from the residual distribution ([ritwork] "Как разреженный
черновик сохраняет ответы плотной модели").  The acceptance rule is the
standard one for exact speculative sampling:

  for i = 1..k:  accept x_i with probability min(1, p_i(x_i) / q_i(x_i))
  first rejection at i: emit y ~ normalize(max(0, p_i - q_i)), stop
  all k accepted: emit a bonus token y ~ p_{k+1}

Readings where the pages are silent:
  * temperature 1 over the full vocabulary: p_i = softmax(p_logits[i]),
    q_i = softmax(q_logits[i]);
  * accept iff u_i < p_i(x_i) / q_i(x_i) (strict), u_i the Philox uniform of
    (n, i-1, ACCEPT);
  * inverse CDF in token-id order: with r the residual (or p_{k+1}) and C its
    inclusive prefix sums, emit the smallest j with C_j > u * C_last, u the
    Philox uniform of (n, i-1, RESAMPLE) (i-1 = k for the bonus);
  * a residual that sums to zero (p == q in floating point) falls back to p_i.

Parity status: pinned by tests/test_oracle_spec_sample.py: the exactness
theorem itself (chi-square of every emitted position against p_i over 10^6
draws), the closed-form acceptance rate sum_x min(p(x), q(x)), and the special
cases q = p (never reject) and disjoint supports (always reject, emit from p).
"""

import numpy as np

from .philox import philox_uniform, STREAM_ACCEPT, STREAM_RESAMPLE


def _softmax(logits):
    x = np.asarray(logits, dtype=np.float64)
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def residual_row(p_row_logits, q_row_logits):
    """max(0, p - q) for one position (float64), with the p fallback when the
    residual sums to zero."""
    p = _softmax(p_row_logits)
    q = _softmax(q_row_logits)
    r = np.maximum(p - q, 0.0)
    if not r.sum() > 0.0:
        return p
    return r


def spec_sample(p_logits, q_logits, draft_tokens, seed, offset=0, seq_ids=None):
    """Exact speculative sampling of N independent drafted blocks.

    p_logits     [N or 1][k+1][V] target logits for positions 1..k+1
    q_logits     [N or 1][k][V]   draft logits for positions 1..k
    draft_tokens [N][k]           drafted tokens x_1..x_k
    seq_ids      [N] sequence indices used as the Philox counter's first word
                 (default 0..N-1; a subset of a larger batch keeps its ids)
    returns out_tokens [N][k+1] int64 (accepted drafts, then the correcting or
            bonus token, then -1 padding), n_accepted [N] int64, and a dict of
            the intermediate quantities (ratios, uniforms, residual totals)
            used by tests to account for floating-point ties.
    """
    x = np.asarray(draft_tokens, dtype=np.int64)
    N, k = x.shape
    p = _softmax(p_logits)
    q = _softmax(q_logits)
    pn = np.arange(N) if p.shape[0] == N else np.zeros(N, dtype=np.int64)
    qn = np.arange(N) if q.shape[0] == N else np.zeros(N, dtype=np.int64)
    n = np.arange(N)
    cn = n if seq_ids is None else np.asarray(seq_ids, dtype=np.int64)
    pos = np.arange(k)

    px = p[pn[:, None], pos[None, :], x]
    qx = q[qn[:, None], pos[None, :], x]
    with np.errstate(divide="ignore"):
        ratio = px / qx
    u_acc = philox_uniform(seed, offset, cn[:, None], pos[None, :], STREAM_ACCEPT)
    accepted = u_acc < ratio
    if k == 0:
        n_acc = np.zeros(N, dtype=np.int64)
    else:
        n_acc = np.where(accepted.all(axis=1), k, np.argmin(accepted, axis=1))

    # Row to sample from: residual at the first rejection, else p_{k+1}.
    rej = n_acc < k
    row = np.empty((N, p.shape[2]))
    row[~rej] = p[pn[~rej], k]
    if rej.any():
        i = n_acc[rej]
        r = np.maximum(p[pn[rej], i] - q[qn[rej], i], 0.0)
        empty = ~(r.sum(axis=1) > 0.0)
        r[empty] = p[pn[rej][empty], i[empty]]
        row[rej] = r
    cdf = np.cumsum(row, axis=1)
    total = cdf[:, -1]
    u_res = philox_uniform(seed, offset, cn, n_acc, STREAM_RESAMPLE)
    target = u_res * total
    y = np.argmax(cdf > target[:, None], axis=1)

    out = np.full((N, k + 1), -1, dtype=np.int64)
    for j in range(k):
        keep = n_acc > j
        out[keep, j] = x[keep, j]
    out[n, n_acc] = y
    details = {
        "ratio": ratio,
        "u_accept": u_acc,
        "u_resample": u_res,
        "residual_total": total,
        "target": target,
    }
    return out, n_acc.astype(np.int64), details

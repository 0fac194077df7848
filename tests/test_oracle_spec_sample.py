"""Pins for the speculative-sampling oracle.  The pages' claim is that the
output follows the dense policy exactly ([wispaper] "S3R drafts sparsely and
verifies densely"); these tests check that claim statistically on a tiny
vocabulary, plus the closed-form acceptance rate and the degenerate cases."""

import numpy as np
from scipy import special, stats

from oracle import spec_sample

N_DRAWS = 1_000_000


def _draw_drafts(q_logits, n, seed):
    rng = np.random.default_rng(seed)
    q = special.softmax(q_logits[0], axis=-1)
    k, V = q.shape
    x = np.empty((n, k), dtype=np.int64)
    for i in range(k):
        x[:, i] = rng.choice(V, size=n, p=q[i])
    return x


def _chi2_position(out, n_acc, p, j):
    """Emitted token at block position j (exists when n_acc >= j) ~ p_j."""
    have = n_acc >= j
    counts = np.bincount(out[have, j], minlength=p.shape[1])
    expected = p[j] * have.sum()
    keep = expected > 0
    assert counts[~keep].sum() == 0
    return stats.chisquare(counts[keep], expected[keep]).pvalue, have.sum()


def _run(p_logits, q_logits, seed):
    x = _draw_drafts(q_logits, N_DRAWS, seed)
    out, n_acc, det = spec_sample(p_logits, q_logits, x, seed=seed, offset=5)
    return x, out, n_acc, det


def test_output_distribution_equals_target():
    rng = np.random.default_rng(1)
    k, V = 3, 12
    p_logits = rng.normal(0, 1.5, size=(1, k + 1, V))
    q_logits = p_logits[:, :k] + rng.normal(0, 1.0, size=(1, k, V))
    x, out, n_acc, det = _run(p_logits, q_logits, 11)
    p = special.softmax(p_logits[0], axis=-1)
    q = special.softmax(q_logits[0], axis=-1)
    for j in range(k + 1):
        pval, n = _chi2_position(out, n_acc, p, j)
        assert n > 10_000
        assert pval > 1e-3, (j, pval)
    # Closed form: P(accept position 1) = sum_x min(p_1(x), q_1(x)).
    alpha = np.minimum(p[0], q[0]).sum()
    rate = (n_acc >= 1).mean()
    assert abs(rate - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / N_DRAWS)
    # Accepted drafts are copied verbatim, padding is -1.
    for j in range(k):
        keep = n_acc > j
        assert np.array_equal(out[keep, j], x[keep, j])
    assert (out[np.arange(k + 1)[None, :] > n_acc[:, None]] == -1).all()


def test_draft_far_from_target():
    rng = np.random.default_rng(2)
    k, V = 3, 10
    p_logits = rng.normal(0, 1.0, size=(1, k + 1, V))
    q_logits = p_logits[:, :k].copy()
    q_logits[..., :4] += 3.0            # q concentrated on a few tokens
    x, out, n_acc, _ = _run(p_logits, q_logits, 12)
    p = special.softmax(p_logits[0], axis=-1)
    for j in range(k + 1):
        pval, _ = _chi2_position(out, n_acc, p, j)
        assert pval > 1e-3, (j, pval)


def test_q_equals_p_never_rejects():
    rng = np.random.default_rng(3)
    k, V = 3, 9
    p_logits = rng.normal(0, 1.0, size=(1, k + 1, V))
    q_logits = p_logits[:, :k].copy()
    x, out, n_acc, _ = _run(p_logits, q_logits, 13)
    assert (n_acc == k).all()
    p = special.softmax(p_logits[0], axis=-1)
    pval, _ = _chi2_position(out, n_acc, p, k)
    assert pval > 1e-3


def test_disjoint_support_always_rejects_and_emits_from_target():
    k, V = 2, 8
    p_logits = np.zeros((1, k + 1, V))
    p_logits[:, :, 4:] = -1e4           # p lives on tokens 0..3
    q_logits = np.zeros((1, k, V))
    q_logits[:, :, :4] = -1e4           # q lives on tokens 4..7
    x, out, n_acc, _ = _run(p_logits, q_logits, 14)
    assert (n_acc == 0).all()
    counts = np.bincount(out[:, 0], minlength=V)
    assert counts[4:].sum() == 0
    assert stats.chisquare(counts[:4]).pvalue > 1e-3


# ---------------------------------------------------------------- residual_row
# residual_row is the row the oracle resamples from after a rejection, and the
# GPU parity tests use it to judge inverse-CDF ties.  Its pins: the residual of
# disjoint supports is p itself; p = q falls back to p; the closed form
# sum_v max(0, p - q) = 1 - sum_v min(p, q) (the rejection probability); and
# the residual's support is exactly {v : p(v) > q(v)}.

def test_residual_of_disjoint_supports_is_the_target():
    from oracle import residual_row
    p_logits = np.array([0.0, 1.0, -1e4, -1e4, 0.5])
    q_logits = np.array([-1e4, -1e4, 0.0, 2.0, -1e4])
    p = special.softmax(p_logits)
    r = residual_row(p_logits, q_logits)
    np.testing.assert_allclose(r, p, rtol=0, atol=1e-15)


def test_residual_of_equal_rows_falls_back_to_the_target():
    from oracle import residual_row
    x = np.random.default_rng(21).normal(0, 2.0, size=37)
    np.testing.assert_allclose(residual_row(x, x), special.softmax(x), rtol=0, atol=1e-15)


def test_residual_total_is_the_rejection_probability():
    from oracle import residual_row
    rng = np.random.default_rng(22)
    for V in (2, 9, 1000):
        p_logits = rng.normal(0, 3.0, size=V)
        q_logits = p_logits + rng.normal(0, 1.0, size=V)
        p, q = special.softmax(p_logits), special.softmax(q_logits)
        r = residual_row(p_logits, q_logits)
        assert abs(r.sum() - (1.0 - np.minimum(p, q).sum())) < 1e-12
        assert np.all(r >= 0.0)
        # support: positive exactly where the target outweighs the draft
        assert np.array_equal(r > 0.0, p > q)

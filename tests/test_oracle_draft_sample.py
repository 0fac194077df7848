"""Pins for the draft-token oracle: closed forms and the distribution."""

import numpy as np
from scipy import special, stats

from oracle import sample_draft_tokens, philox_uniform, STREAM_DRAFT, STREAM_RESAMPLE


def test_uniform_logits_give_floor_u_times_v():
    # q = 1/V for every token: C_v = (v+1)/V, so the draw is floor(u * V).
    for V in (1, 7, 64, 1000):
        ids = np.arange(5000)
        tok, det = sample_draft_tokens(np.zeros((1, V)), seed=3, offset=1, draft_pos=2, seq_ids=ids)
        u = philox_uniform(3, 1, ids, 2, STREAM_DRAFT)
        np.testing.assert_array_equal(tok, np.floor(u * V).astype(np.int64))


def test_dominant_logit_is_always_drawn():
    logits = np.zeros((50, 300))
    logits[np.arange(50), np.arange(50) * 5] = 1000.0
    tok, _ = sample_draft_tokens(logits, seed=9, offset=0, draft_pos=0)
    np.testing.assert_array_equal(tok, np.arange(50) * 5)


def test_draws_follow_softmax():
    rng = np.random.default_rng(4)
    V = 16
    logits = rng.normal(0, 1.5, size=(1, V))
    N = 1_000_000
    tok, _ = sample_draft_tokens(logits, seed=21, offset=5, draft_pos=3, seq_ids=np.arange(N))
    q = special.softmax(logits[0])
    counts = np.bincount(tok, minlength=V)
    assert stats.chisquare(counts, q * N).pvalue > 1e-3


def test_draft_stream_is_its_own():
    ids = np.arange(1000)
    assert not np.array_equal(philox_uniform(1, 0, ids, 0, STREAM_DRAFT), philox_uniform(1, 0, ids, 0, STREAM_RESAMPLE))

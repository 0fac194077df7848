"""Pins for the scheduler oracle: the AIMD limit's additive ramp and
multiplicative cut in closed form, a trace worked out by hand on a 4-request
pool, conservation and pool invariants on random workloads, the restore-first
priority, a pool that never fills, and offload and recompute taking the same
decisions."""

import math

import pytest

from oracle.scheduler import (POLICY_AIMD, POLICY_FIXED_OFFLOAD, POLICY_RECOMPUTE, simulate)
from workloads import make_rollout_requests


def _cfg(policy, pool, **over):
    c = dict(policy=policy, pool_pages=pool, page_size=16, block_tokens=5, limit_init=64, limit_min=8,
             limit_max=512, add_step=8, mult=0.5, util_low=0.8, util_high=0.95, backlog_max=0)
    c.update(over)
    return c


def _long(n, response=100_000):
    return [10] * n, [response] * n, [[1]] * n


def test_additive_ramp_closed_form():
    cfg = _cfg(POLICY_AIMD, 10**9, limit_init=2, add_step=3, limit_max=20, util_low=0.5)
    tot, trace = simulate(cfg, *_long(50), max_steps=10)
    assert [t["limit"] for t in trace] == [min(20, 2 + 3 * t) for t in range(1, 11)]
    assert [t["ran"] for t in trace] == [min(20, 2 + 3 * (t - 1)) for t in range(1, 11)]
    assert tot["tokens"] == sum(min(20, 2 + 3 * (t - 1)) for t in range(1, 11))


def test_multiplicative_cut_closed_form():
    """backlog_max = -1: every step counts as backlogged; the limit halves down
    to limit_min.  The limit gates admission only, so the 64 requests admitted
    at the start keep running."""
    cfg = _cfg(POLICY_AIMD, 10**9, limit_init=64, limit_min=3, mult=0.5, backlog_max=-1)
    tot, trace = simulate(cfg, *_long(100), max_steps=8)
    want, lim = [], 64
    for _ in range(8):
        lim = max(3, math.floor(lim * 0.5))
        want.append(lim)
    assert [t["limit"] for t in trace] == want == [32, 16, 8, 4, 3, 3, 3, 3]
    assert all(t["ran"] == 64 for t in trace) and trace[0]["admitted"] == 64


@pytest.mark.parametrize("policy", [POLICY_FIXED_OFFLOAD, POLICY_RECOMPUTE])
def test_hand_worked_trace(policy):
    """Pool of 6 pages of 4 tokens, block 2, limit 3; requests (P, T):
    (3, 4), (5, 3), (2, 6), (1, 2); every round emits 2.
    Step 1: admit r0 (2 pages), r1 (2), r2 (1); r3 waits (limit).  Round:
            g = 2, 2, 2.  Reserved 5.
    Step 2: r1 grows to 3 pages (free 0); r2 needs 2 pages, no later request
            to pause, so r2 pauses itself (1 page offloaded / dropped).
            Round: r0 and r1 finish (r1 emits only 1).  Reserved 5, used 0.
    Step 3: restore r2 first (2 pages; offload moves its 1 host page back,
            recompute recomputes ceil(4/4) = 1 page), then admit r3 (1 page).
            Round: r2 -> 4, r3 finishes.  Reserved 3, used 2.
    Step 4: r2 finishes.  Reserved 2, used 0."""
    cfg = _cfg(policy, 6, page_size=4, block_tokens=2, limit_init=3)
    tot, trace = simulate(cfg, [3, 5, 2, 1], [4, 3, 6, 2], [[2], [2], [2], [2]])
    assert [(t["ran"], t["admitted"], t["resumed"], t["paused"], t["reserved"], t["used"]) for t in trace] == \
        [(3, 3, 0, 0, 5, 5), (2, 0, 0, 1, 5, 0), (2, 1, 1, 0, 3, 2), (1, 0, 0, 0, 2, 0)]
    assert tot["steps"] == 4 and tot["tokens"] == 15 and tot["preemptions"] == 1 and tot["peak_used"] == 5
    assert tot["running_sum"] == 8
    if policy == POLICY_FIXED_OFFLOAD:
        assert (tot["offloaded"], tot["restored"], tot["dropped"], tot["recomputed"]) == (1, 1, 0, 0)
        assert [t["moved"] for t in trace] == [0, 1, 1, 0]
    else:
        assert (tot["offloaded"], tot["restored"], tot["dropped"], tot["recomputed"]) == (0, 0, 1, 1)


@pytest.mark.parametrize("policy", [POLICY_AIMD, POLICY_FIXED_OFFLOAD, POLICY_RECOMPUTE])
@pytest.mark.parametrize("seed", [1, 2])
def test_invariants_on_random_workloads(policy, seed):
    w = make_rollout_requests(12, 4, seed, prompt_lo=64, prompt_hi=256, response_lo=64, response_hi=2048)
    pool = 400                                   # tight: forces pauses
    cfg = _cfg(policy, pool, limit_init=24, limit_min=2, limit_max=48, add_step=2, util_low=0.6, util_high=0.9,
               backlog_max=2)
    tot, trace = simulate(cfg, w.prompt_lens, w.response_lens, w.emits)
    assert not tot["stalled"]
    assert tot["tokens"] == int(w.response_lens.sum())
    assert tot["preemptions"] > 0
    assert all(t["reserved"] <= pool and t["used"] <= pool for t in trace)
    if policy != POLICY_RECOMPUTE:
        assert tot["restored"] == tot["offloaded"] and tot["dropped"] == tot["recomputed"] == 0
    else:
        assert tot["offloaded"] == tot["restored"] == 0 and tot["recomputed"] > 0
    assert sum(t["moved"] for t in trace) == tot["offloaded"] + tot["restored"]
    # restore first: a new request is admitted only once no paused request is left
    prev_paused = 0
    for t in trace:
        if t["admitted"] > 0:
            assert t["resumed"] == prev_paused
        prev_paused = t["paused"]
    if policy != POLICY_AIMD:
        assert all(t["limit"] == 24 for t in trace)


def test_pool_that_never_fills_moves_nothing():
    w = make_rollout_requests(8, 4, 3, prompt_lo=64, prompt_hi=256, response_lo=64, response_hi=2048)
    for policy in (POLICY_AIMD, POLICY_FIXED_OFFLOAD, POLICY_RECOMPUTE):
        tot, _ = simulate(_cfg(policy, 10**7, limit_init=16, limit_min=2), w.prompt_lens, w.response_lens,
                          w.emits)
        assert tot["preemptions"] == tot["offloaded"] == tot["restored"] == tot["dropped"] == tot["recomputed"] == 0
        assert tot["tokens"] == int(w.response_lens.sum())


def test_offload_and_recompute_take_the_same_decisions():
    w = make_rollout_requests(10, 4, 5, prompt_lo=64, prompt_hi=256, response_lo=64, response_hi=2048)
    off, t_off = simulate(_cfg(POLICY_FIXED_OFFLOAD, 300, limit_init=20), w.prompt_lens, w.response_lens, w.emits)
    rec, t_rec = simulate(_cfg(POLICY_RECOMPUTE, 300, limit_init=20), w.prompt_lens, w.response_lens, w.emits)
    keys = ("ran", "admitted", "resumed", "limit", "paused", "reserved", "used")
    assert [tuple(t[k] for k in keys) for t in t_off] == [tuple(t[k] for k in keys) for t in t_rec]
    assert off["offloaded"] == rec["dropped"] > 0 and off["steps"] == rec["steps"]


def test_stall_when_a_request_exceeds_the_pool():
    tot, trace = simulate(_cfg(POLICY_FIXED_OFFLOAD, 4, page_size=4), [100], [10], [[1]])
    assert tot["stalled"] == 1 and tot["steps"] == 0 and trace == []

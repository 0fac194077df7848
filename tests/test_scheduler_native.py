"""The library's C++ scheduler against the oracle: identical totals and
identical per-step records (every field is an integer, and the one ratio and
the one product are taken in double on both sides) on random rollout
workloads, for the three policies and several pool sizes; the step-by-step
handle reports the requests of each round; bad configurations are refused.
Host code only: runs without a GPU."""

import numpy as np
import pytest

from oracle.scheduler import simulate
from speculative_decode_attention_paged_b300 import S3RError
from speculative_decode_attention_paged_b300 import scheduler as sched
from workloads import make_rollout_requests


def _cfg(policy, pool, **over):
    c = dict(policy=policy, pool_pages=pool, page_size=16, block_tokens=5, limit_init=24, limit_min=2,
             limit_max=64, add_step=2, mult=0.5, util_low=0.6, util_high=0.9, backlog_max=2)
    c.update(over)
    return c


@pytest.mark.parametrize("policy", [sched.AIMD, sched.FIXED_OFFLOAD, sched.RECOMPUTE])
@pytest.mark.parametrize("pool", [250, 400, 900, 10**6])
def test_native_equals_oracle(policy, pool):
    w = make_rollout_requests(12, 4, pool % 97, prompt_lo=64, prompt_hi=256, response_lo=64, response_hi=2048)
    cfg = _cfg(policy, pool)
    ref_tot, ref_trace = simulate(cfg, w.prompt_lens, w.response_lens, w.emits)
    tot, trace = sched.run(cfg, w.prompt_lens, w.response_lens, w.emits)
    assert tot == {k: ref_tot[k] for k in tot}
    assert trace == ref_trace


def test_native_equals_oracle_with_odd_constants():
    w = make_rollout_requests(20, 8, 11, prompt_lo=16, prompt_hi=300, response_lo=8, response_hi=900, k=6,
                              alpha=0.55)
    cfg = _cfg(sched.AIMD, 333, page_size=7, block_tokens=7, limit_init=10, limit_min=3, limit_max=37, add_step=5,
               mult=0.7, util_low=0.45, util_high=0.77, backlog_max=5)
    ref_tot, ref_trace = simulate(cfg, w.prompt_lens, w.response_lens, w.emits)
    tot, trace = sched.run(cfg, w.prompt_lens, w.response_lens, w.emits)
    assert tot == {k: ref_tot[k] for k in tot} and trace == ref_trace


def test_step_handle_reports_each_round():
    w = make_rollout_requests(6, 4, 7, prompt_lo=64, prompt_hi=256, response_lo=64, response_hi=1024)
    cfg = _cfg(sched.AIMD, 300)
    s = sched.Scheduler(cfg, w.prompt_lens, w.response_lens, w.emits)
    ref_tot, ref_trace = simulate(cfg, w.prompt_lens, w.response_lens, w.emits)
    seen, recs = np.zeros(w.n, dtype=np.int64), []
    while not s.finished:
        rec, ids = s.step()
        recs.append(rec)
        assert len(ids) == rec["ran"] and len(set(ids.tolist())) == len(ids)
        seen[ids] += 1
    assert recs == ref_trace
    assert s.totals() == {k: ref_tot[k] for k in s.totals()}
    assert seen.sum() == ref_tot["running_sum"] and np.all(seen > 0)
    rec, ids = s.step()                        # after the end: nothing happens
    assert rec["ran"] == 0 and len(ids) == 0
    s.close()


def test_stall_is_reported():
    tot, trace = sched.run(_cfg(sched.FIXED_OFFLOAD, 4, page_size=4), [100], [10], [[1]])
    assert tot["stalled"] == 1 and tot["steps"] == 0 and trace == []


@pytest.mark.parametrize("over", [dict(pool_pages=0), dict(page_size=0), dict(block_tokens=0), dict(limit_init=0),
                                  dict(policy=3), dict(mult=0.0), dict(mult=1.5), dict(limit_min=30),
                                  dict(limit_max=10), dict(util_low=0.95, util_high=0.9)])
def test_bad_configurations_are_refused(over):
    cfg = _cfg(sched.AIMD, 100)
    cfg.update(over)
    with pytest.raises(S3RError):
        sched.run(cfg, [10], [10], [[1]])


def test_bad_requests_are_refused():
    cfg = _cfg(sched.AIMD, 100)
    for args in (([10], [0], [[1]]), ([-1], [5], [[1]]), ([10], [5], [[0]]), ([10], [5], [[]])):
        with pytest.raises(S3RError):
            sched.run(cfg, *args)

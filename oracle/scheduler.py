"""Oracle for the KV-aware AIMD rollout scheduler, simulated over a page pool.

Test infrastructure only (see the package docstring).

What the pages fix
------------------
* Dense verification needs each request's complete history in GPU memory, so
  under memory pressure KV pages are offloaded to the host and restored later;
  pages that go out and come back repeatedly (thrashing) cost transfer time
  ([wispaper] "Dense verification still pays the full KV-cache bill").
* The scheduler adapts request admission by AIMD: GPU KV utilisation measures
  resident pressure and a restoration backlog records the outstanding demand
  of paused requests; under low utilisation the concurrency limit rises by an
  additive step, and high utilisation or an excessive backlog cuts it
  multiplicatively ([wispaper] same section; [rebas] "真正难搬的，还是那叠完整笔记").
* Paused requests keep their token and proposal state and are restored
  first ([wispaper]; [rebas] same section: paused requests are restored with
  priority).
* Baselines: offload with a fixed concurrency limit of 256, and recompute
  (evicted prefixes are recomputed instead of moved).  Reported: cache pages
  moved per 1000 generated tokens; cumulative recompute and moved pages
  ([rebas] same section; [wispaper] "What to watch").

Readings where the pages are silent
-----------------------------------
* One scheduler step is one S³R round of every running request.  Before the
  round each running request holds pages for its context plus the k + 1
  tokens the round may write: pages_for(P + g + k + 1), pages of 16 tokens.
* A step admits first, then runs the round, then updates the limit.
* Growth is served in admission order; when the pool is short, the most
  recently admitted other running request is paused (LIFO), and if none is
  left the request itself is paused.  Offload policies move a paused
  request's resident pages to the host (counted as moved); the recompute
  policy drops them.
* The round then emits, for each running request, the next entry of its
  emitted-token sequence (accepted drafts + 1), capped at its response length;
  a finished request frees its pages.
* AIMD (after the round, finished requests' pages freed): util = used pages /
  pool pages, backlog = number of
  paused requests; util > util_high or backlog > backlog_max cuts the limit
  to max(limit_min, floor(limit * mult)); else util < util_low raises it to
  min(limit_max, limit + add_step).  The fixed policies keep limit_init.
* Admission (at the start of the next step), while fewer than `limit`
  requests run: the
  oldest paused request if its pages fit (restoring moves its host pages
  back, or for recompute recomputes pages_for(P + g)), else stop; when none
  is paused, the next waiting request if pages_for(P + k + 1) fit (its
  prefill is not a move), else stop.

Parity status: pinned by tests/test_oracle_scheduler.py: the additive ramp
and the multiplicative cut in closed form, a hand-worked trace on a 3-request
pool, conservation of tokens, pages never above the pool, restored = offloaded
at the end, a pool that never fills moves nothing, and offload and recompute
taking identical decisions with moved pages = dropped + recomputed.
"""

import math

POLICY_AIMD, POLICY_FIXED_OFFLOAD, POLICY_RECOMPUTE = 0, 1, 2
WAITING, RUNNING, PAUSED, DONE = 0, 1, 2, 3


def pages_for(tokens, page_size):
    return -(-int(tokens) // int(page_size))


def simulate(cfg, prompt_lens, response_lens, emits, max_steps=1_000_000):
    """Run the scheduler to completion.

    cfg            dict: policy, pool_pages, page_size, block_tokens (k + 1),
                   limit_init, limit_min, limit_max, add_step, mult, util_low,
                   util_high, backlog_max
    prompt_lens    [R] prompt tokens; response_lens [R] tokens to generate
    emits          list of R sequences: tokens emitted by each of the
                   request's rounds (accepted drafts + 1)
    returns (totals dict, per-step list of dicts)
    """
    R = len(prompt_lens)
    ps, blk = int(cfg["page_size"]), int(cfg["block_tokens"])
    pool = int(cfg["pool_pages"])
    policy = int(cfg["policy"])
    limit = int(cfg["limit_init"])
    status = [WAITING] * R
    gen = [0] * R
    rounds = [0] * R
    gpu = [0] * R
    host = [0] * R
    waiting = list(range(R))
    running, paused = [], []
    free = pool
    tot = {"steps": 0, "tokens": 0, "offloaded": 0, "restored": 0, "dropped": 0, "recomputed": 0,
           "preemptions": 0, "peak_used": 0, "running_sum": 0, "stalled": 0}
    trace = []

    def evict(v):
        nonlocal free
        if policy == POLICY_RECOMPUTE:
            tot["dropped"] += gpu[v]
        else:
            tot["offloaded"] += gpu[v]
            host[v] = gpu[v]
        free += gpu[v]
        gpu[v] = 0
        status[v] = PAUSED
        paused.append(v)
        tot["preemptions"] += 1

    while (waiting or running or paused) and tot["steps"] < max_steps:
        step_moved = tot["offloaded"] + tot["restored"]
        admitted = resumed = 0
        # (1) admission: paused requests first, then new ones
        while len(running) < limit:
            if paused:
                r = paused[0]
                need = pages_for(prompt_lens[r] + gen[r] + blk, ps)
                if need > free:
                    break
                paused.pop(0)
                resumed += 1
                if policy == POLICY_RECOMPUTE:
                    tot["recomputed"] += pages_for(prompt_lens[r] + gen[r], ps)
                else:
                    tot["restored"] += host[r]
                    host[r] = 0
            elif waiting:
                r = waiting[0]
                need = pages_for(prompt_lens[r] + blk, ps)
                if need > free:
                    break
                waiting.pop(0)
                admitted += 1
            else:
                break
            free -= need
            gpu[r] = need
            status[r] = RUNNING
            running.append(r)
        if not running:
            tot["stalled"] = 1          # nothing runs and nothing can be admitted
            break
        # (2) every running request reserves the pages of this round
        i = 0
        while i < len(running):
            r = running[i]
            need = pages_for(prompt_lens[r] + gen[r] + blk, ps) - gpu[r]
            while need > free and len(running) - 1 > i:
                evict(running.pop())
            if need > free:
                running.pop(i)
                evict(r)
                continue
            if need > 0:
                free -= need
                gpu[r] += need
            i += 1
        reserved = pool - free
        tot["peak_used"] = max(tot["peak_used"], reserved)
        ctx = sum(int(prompt_lens[r]) + gen[r] for r in running)
        # (3) the round
        still = []
        for r in running:
            e = emits[r][rounds[r]] if rounds[r] < len(emits[r]) else emits[r][-1]
            e = min(int(e), int(response_lens[r]) - gen[r])
            gen[r] += e
            rounds[r] += 1
            tot["tokens"] += e
            if gen[r] >= response_lens[r]:
                status[r] = DONE
                free += gpu[r]
                gpu[r] = 0
            else:
                still.append(r)
        n_ran = len(running)
        tot["running_sum"] += n_ran
        running = still
        used = pool - free
        # (4) AIMD update of the concurrency limit
        if policy == POLICY_AIMD:
            util = used / pool
            if util > cfg["util_high"] or len(paused) > cfg["backlog_max"]:
                limit = max(int(cfg["limit_min"]), int(math.floor(limit * cfg["mult"])))
            elif util < cfg["util_low"]:
                limit = min(int(cfg["limit_max"]), limit + int(cfg["add_step"]))
        tot["steps"] += 1
        trace.append({"ran": n_ran, "admitted": admitted, "resumed": resumed, "limit": limit,
                      "paused": len(paused), "reserved": reserved, "used": used, "ctx_tokens": ctx,
                      "moved": tot["offloaded"] + tot["restored"] - step_moved})
    tot["limit_final"] = limit
    return tot, trace

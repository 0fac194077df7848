// KV-aware AIMD rollout scheduler over a page pool (host code).
//
// The S³R pages: dense verification keeps every running request's whole KV
// history on the GPU; under memory pressure pages are offloaded and restored,
// and the scheduler adapts admission by additive increase / multiplicative
// decrease on GPU KV utilisation and the restoration backlog, restoring
// paused requests first (wispaper.ai, "Dense verification still pays the full
// KV-cache bill"; rebasdaily.com, "真正难搬的，还是那叠完整笔记").  The step
// rules are stated in include/s3r_sched.h.
//
// State is per request (status, generated tokens, rounds, resident and host
// pages) plus three queues: waiting (FIFO by id), running (admission order)
// and paused (FIFO by pause time).  All arithmetic is integer except the
// utilisation ratio and the multiplicative cut, taken in double.

#include <cmath>
#include <cstdint>
#include <deque>
#include <new>
#include <vector>

#include "../../include/s3r_sched.h"

struct s3r_sched {
  s3r_sched_config cfg;
  std::vector<int32_t> prompt, response;
  std::vector<int64_t> emit_off;
  std::vector<int32_t> emits;
  std::vector<int32_t> status, gen, rounds;
  std::vector<int64_t> gpu, host;
  std::deque<int32_t> waiting, paused;
  std::vector<int32_t> running;
  int64_t free_pages = 0;
  int32_t limit = 0;
  int32_t finished = 0;
  s3r_sched_totals tot{};
};

namespace {

enum : int32_t { kWaiting = 0, kRunning = 1, kPaused = 2, kDone = 3 };

int64_t pages_for(int64_t tokens, int32_t page_size) { return (tokens + page_size - 1) / page_size; }

bool valid_config(const s3r_sched_config* c) {
  if (c == nullptr) return false;
  if (c->policy < S3R_SCHED_AIMD || c->policy > S3R_SCHED_RECOMPUTE) return false;
  if (c->pool_pages <= 0 || c->page_size <= 0 || c->block_tokens < 1) return false;
  if (c->limit_init < 1 || c->add_step < 0) return false;
  if (c->policy == S3R_SCHED_AIMD) {
    if (c->limit_min < 1 || c->limit_min > c->limit_init || c->limit_init > c->limit_max) return false;
    if (!(c->mult > 0.0 && c->mult <= 1.0)) return false;
    if (!(c->util_low <= c->util_high)) return false;
  }
  return true;
}

void evict(s3r_sched* s, int32_t v) {
  if (s->cfg.policy == S3R_SCHED_RECOMPUTE) {
    s->tot.dropped += s->gpu[v];
  } else {
    s->tot.offloaded += s->gpu[v];
    s->host[v] = s->gpu[v];
  }
  s->free_pages += s->gpu[v];
  s->gpu[v] = 0;
  s->status[v] = kPaused;
  s->paused.push_back(v);
  ++s->tot.preemptions;
}

int32_t emit_of(const s3r_sched* s, int32_t r) {
  const int64_t lo = s->emit_off[r], hi = s->emit_off[r + 1];
  const int64_t i = lo + s->rounds[r];
  return s->emits[i < hi ? i : hi - 1];
}

}  // namespace

extern "C" {

s3r_status s3r_sched_create(const s3r_sched_config* cfg, int32_t n, const int32_t* prompt_lens,
                            const int32_t* response_lens, const int64_t* emit_offsets, const int32_t* emits,
                            s3r_sched** out) {
  if (out == nullptr) return S3R_ERR_INVALID_ARG;
  *out = nullptr;
  if (!valid_config(cfg) || n < 0) return S3R_ERR_INVALID_ARG;
  if (n > 0 && (prompt_lens == nullptr || response_lens == nullptr || emit_offsets == nullptr || emits == nullptr))
    return S3R_ERR_INVALID_ARG;
  if (n > 0 && emit_offsets[0] != 0) return S3R_ERR_INVALID_ARG;
  for (int32_t r = 0; r < n; ++r) {
    if (prompt_lens[r] < 0 || response_lens[r] < 1) return S3R_ERR_INVALID_ARG;
    if (emit_offsets[r + 1] <= emit_offsets[r]) return S3R_ERR_INVALID_ARG;
    for (int64_t i = emit_offsets[r]; i < emit_offsets[r + 1]; ++i)
      if (emits[i] < 1) return S3R_ERR_INVALID_ARG;
  }
  s3r_sched* s = new (std::nothrow) s3r_sched();
  if (s == nullptr) return S3R_ERR_INVALID_ARG;
  s->cfg = *cfg;
  s->prompt.assign(prompt_lens, prompt_lens + n);
  s->response.assign(response_lens, response_lens + n);
  s->emit_off.assign(emit_offsets, emit_offsets + n + 1);
  if (n == 0) s->emit_off.assign(1, 0);
  s->emits.assign(emits, emits + s->emit_off.back());
  s->status.assign(n, kWaiting);
  s->gen.assign(n, 0);
  s->rounds.assign(n, 0);
  s->gpu.assign(n, 0);
  s->host.assign(n, 0);
  for (int32_t r = 0; r < n; ++r) s->waiting.push_back(r);
  s->free_pages = cfg->pool_pages;
  s->limit = cfg->limit_init;
  s->finished = n == 0 ? 1 : 0;
  *out = s;
  return S3R_OK;
}

s3r_status s3r_sched_step(s3r_sched* s, s3r_sched_step_record* rec, int32_t* ran_ids, int32_t capacity,
                          int32_t* n_ran, int32_t* finished) {
  if (s == nullptr || (ran_ids != nullptr && capacity < 0)) return S3R_ERR_INVALID_ARG;
  s3r_sched_step_record r{};
  if (n_ran != nullptr) *n_ran = 0;
  if (s->finished) {
    if (rec != nullptr) *rec = r;
    if (finished != nullptr) *finished = 1;
    return S3R_OK;
  }
  const s3r_sched_config& c = s->cfg;
  const int32_t ps = c.page_size, blk = c.block_tokens;
  const int64_t moved_before = s->tot.offloaded + s->tot.restored;
  // 1. admission: paused requests first, then new ones
  while (static_cast<int64_t>(s->running.size()) < s->limit) {
    int32_t q;
    int64_t need;
    if (!s->paused.empty()) {
      q = s->paused.front();
      need = pages_for(static_cast<int64_t>(s->prompt[q]) + s->gen[q] + blk, ps);
      if (need > s->free_pages) break;
      s->paused.pop_front();
      ++r.resumed;
      if (c.policy == S3R_SCHED_RECOMPUTE) {
        s->tot.recomputed += pages_for(static_cast<int64_t>(s->prompt[q]) + s->gen[q], ps);
      } else {
        s->tot.restored += s->host[q];
        s->host[q] = 0;
      }
    } else if (!s->waiting.empty()) {
      q = s->waiting.front();
      need = pages_for(static_cast<int64_t>(s->prompt[q]) + blk, ps);
      if (need > s->free_pages) break;
      s->waiting.pop_front();
      ++r.admitted;
    } else {
      break;
    }
    s->free_pages -= need;
    s->gpu[q] = need;
    s->status[q] = kRunning;
    s->running.push_back(q);
  }
  if (s->running.empty()) {
    s->tot.stalled = 1;            // nothing runs and nothing can be admitted
    s->finished = 1;
    s->tot.limit_final = s->limit;
    if (rec != nullptr) *rec = r;
    if (finished != nullptr) *finished = 1;
    return S3R_OK;
  }
  // 2. every running request reserves the pages of this round
  size_t i = 0;
  while (i < s->running.size()) {
    const int32_t q = s->running[i];
    const int64_t need = pages_for(static_cast<int64_t>(s->prompt[q]) + s->gen[q] + blk, ps) - s->gpu[q];
    while (need > s->free_pages && s->running.size() - 1 > i) {
      const int32_t v = s->running.back();
      s->running.pop_back();
      evict(s, v);
    }
    if (need > s->free_pages) {
      s->running.erase(s->running.begin() + static_cast<std::ptrdiff_t>(i));
      evict(s, q);
      continue;
    }
    if (need > 0) {
      s->free_pages -= need;
      s->gpu[q] += need;
    }
    ++i;
  }
  r.reserved = c.pool_pages - s->free_pages;
  if (r.reserved > s->tot.peak_used) s->tot.peak_used = r.reserved;
  for (const int32_t q : s->running) r.ctx_tokens += static_cast<int64_t>(s->prompt[q]) + s->gen[q];
  // 3. the round
  r.ran = static_cast<int32_t>(s->running.size());
  if (n_ran != nullptr) *n_ran = r.ran;
  if (ran_ids != nullptr)
    for (int32_t j = 0; j < r.ran && j < capacity; ++j) ran_ids[j] = s->running[j];
  std::vector<int32_t> still;
  still.reserve(s->running.size());
  for (const int32_t q : s->running) {
    int32_t e = emit_of(s, q);
    const int32_t left = s->response[q] - s->gen[q];
    if (e > left) e = left;
    s->gen[q] += e;
    ++s->rounds[q];
    s->tot.tokens += e;
    if (s->gen[q] >= s->response[q]) {
      s->status[q] = kDone;
      s->free_pages += s->gpu[q];
      s->gpu[q] = 0;
    } else {
      still.push_back(q);
    }
  }
  s->tot.running_sum += r.ran;
  s->running.swap(still);
  r.used = c.pool_pages - s->free_pages;
  // 4. AIMD update of the concurrency limit
  if (c.policy == S3R_SCHED_AIMD) {
    const double util = static_cast<double>(r.used) / static_cast<double>(c.pool_pages);
    if (util > c.util_high || static_cast<int64_t>(s->paused.size()) > c.backlog_max) {
      const int32_t cut = static_cast<int32_t>(std::floor(static_cast<double>(s->limit) * c.mult));
      s->limit = cut > c.limit_min ? cut : c.limit_min;
    } else if (util < c.util_low) {
      const int64_t up = static_cast<int64_t>(s->limit) + c.add_step;
      s->limit = static_cast<int32_t>(up < c.limit_max ? up : c.limit_max);
    }
  }
  ++s->tot.steps;
  r.limit = s->limit;
  r.paused = static_cast<int32_t>(s->paused.size());
  r.moved = s->tot.offloaded + s->tot.restored - moved_before;
  if (s->waiting.empty() && s->running.empty() && s->paused.empty()) s->finished = 1;
  s->tot.limit_final = s->limit;
  if (rec != nullptr) *rec = r;
  if (finished != nullptr) *finished = s->finished;
  return S3R_OK;
}

s3r_status s3r_sched_get_totals(const s3r_sched* s, s3r_sched_totals* out) {
  if (s == nullptr || out == nullptr) return S3R_ERR_INVALID_ARG;
  *out = s->tot;
  out->limit_final = s->limit;
  return S3R_OK;
}

void s3r_sched_destroy(s3r_sched* s) { delete s; }

s3r_status s3r_sched_run(const s3r_sched_config* cfg, int32_t n, const int32_t* prompt_lens,
                         const int32_t* response_lens, const int64_t* emit_offsets, const int32_t* emits,
                         int64_t max_steps, s3r_sched_step_record* trace, s3r_sched_totals* out) {
  if (out == nullptr || max_steps < 0) return S3R_ERR_INVALID_ARG;
  s3r_sched* s = nullptr;
  const s3r_status st = s3r_sched_create(cfg, n, prompt_lens, response_lens, emit_offsets, emits, &s);
  if (st != S3R_OK) return st;
  int32_t done = s->finished;
  for (int64_t t = 0; t < max_steps && !done; ++t) {
    s3r_sched_step_record rec{};
    const int64_t before = s->tot.steps;
    s3r_sched_step(s, &rec, nullptr, 0, nullptr, &done);
    if (trace != nullptr && s->tot.steps > before) trace[before] = rec;
  }
  s3r_sched_get_totals(s, out);
  s3r_sched_destroy(s);
  return S3R_OK;
}

}  // extern "C"

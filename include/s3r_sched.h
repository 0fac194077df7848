/*
 * s3r_sched.h — host-side KV-aware AIMD rollout scheduler over a page pool.
 *
 * Dense verification needs every running request's whole KV history on the
 * GPU, so under memory pressure pages are offloaded to the host and restored
 * later, and pages that move back and forth (thrashing) cost transfer time
 * (wispaper.ai, "Dense verification still pays the full KV-cache bill").
 * The scheduler adapts admission by additive increase and multiplicative
 * decrease: GPU KV utilisation measures resident pressure, the restoration
 * backlog the demand of paused requests; low utilisation raises the
 * concurrency limit by a step, high utilisation or an excessive backlog cuts
 * it by a factor; paused requests keep their state and are restored first
 * (wispaper.ai, same section; rebasdaily.com, "真正难搬的，还是那叠完整笔记").
 * The pages print no constants; they are the caller's.  Baselines: offload
 * with a fixed limit, and recompute (evicted prefixes recomputed, not moved).
 *
 * Everything here is host code and host memory; no call touches a GPU.
 *
 * One step is one S³R round of every running request:
 *   1. admission while fewer than `limit` requests run: the oldest paused
 *      request if its pages fit (restoring moves its host pages back, or for
 *      recompute recomputes ceil((P + g) / page_size) pages), else stop; with
 *      none paused, the next waiting request if ceil((P + block) / page_size)
 *      pages fit, else stop;
 *   2. each running request, in admission order, grows to
 *      ceil((P + g + block) / page_size) resident pages; when the pool is
 *      short the most recently admitted other request is paused, and if none
 *      is left the request itself (offload: its pages move to the host;
 *      recompute: they are dropped);
 *   3. the round: each running request emits its next entry of `emits`
 *      (capped at its response length); finished requests free their pages;
 *   4. AIMD only: util = used / pool_pages, backlog = paused requests;
 *      util > util_high or backlog > backlog_max: limit =
 *      max(limit_min, floor(limit * mult)); else util < util_low: limit =
 *      min(limit_max, limit + add_step).
 * P = prompt tokens, g = generated tokens, block = block_tokens (k + 1).
 */
#ifndef S3R_SCHED_H_
#define S3R_SCHED_H_

#include <stdint.h>

#include "s3r.h"

#ifdef __cplusplus
extern "C" {
#endif

#define S3R_SCHED_AIMD 0
#define S3R_SCHED_FIXED_OFFLOAD 1
#define S3R_SCHED_RECOMPUTE 2

typedef struct s3r_sched_config {
  int32_t policy;        /* S3R_SCHED_* */
  int64_t pool_pages;    /* GPU pages for KV (> 0) */
  int32_t page_size;     /* tokens per page (> 0) */
  int32_t block_tokens;  /* tokens a round may write, k + 1 (>= 1) */
  int32_t limit_init;    /* concurrency limit at the start (the fixed policies' limit) */
  int32_t limit_min;     /* AIMD bounds: 1 <= limit_min <= limit_init <= limit_max */
  int32_t limit_max;
  int32_t add_step;      /* additive increase (>= 0) */
  double mult;           /* multiplicative decrease, in (0, 1] */
  double util_low;       /* increase below this utilisation */
  double util_high;      /* decrease above this utilisation */
  int32_t backlog_max;   /* decrease when more requests than this are paused */
} s3r_sched_config;

typedef struct s3r_sched_totals {
  int64_t steps;         /* rounds run */
  int64_t tokens;        /* tokens emitted */
  int64_t offloaded;     /* pages moved GPU -> host */
  int64_t restored;      /* pages moved host -> GPU */
  int64_t dropped;       /* pages dropped (recompute policy) */
  int64_t recomputed;    /* pages recomputed on restore (recompute policy) */
  int64_t preemptions;   /* requests paused */
  int64_t peak_used;     /* most pages reserved in one round */
  int64_t running_sum;   /* sum over rounds of the requests that ran */
  int32_t stalled;       /* 1: nothing could run (a request larger than the pool) */
  int32_t limit_final;
} s3r_sched_totals;

typedef struct s3r_sched_step_record {
  int32_t ran;           /* requests in the round */
  int32_t admitted;      /* new requests admitted before it */
  int32_t resumed;       /* paused requests restored before it */
  int32_t limit;         /* limit after the AIMD update */
  int32_t paused;        /* paused requests after the round */
  int32_t pad;
  int64_t reserved;      /* pages reserved for the round */
  int64_t used;          /* pages in use after the round */
  int64_t moved;         /* pages offloaded + restored in this step */
  int64_t ctx_tokens;    /* sum of P + g over the round's requests, before it */
} s3r_sched_step_record;

typedef struct s3r_sched s3r_sched;   /* opaque */

/*
 * Create a scheduler for n_requests requests (all waiting).  Host arrays,
 * copied: prompt_lens[n] (>= 0), response_lens[n] (>= 1), and the tokens each
 * round of request r emits, emits[emit_offsets[r] .. emit_offsets[r+1]) (each
 * >= 1; rounds past the end repeat the last entry; at least one entry per
 * request).  Writes the handle to *out.  Invalid configurations or arrays
 * return S3R_ERR_INVALID_ARG.
 */
S3R_API s3r_status s3r_sched_create(const s3r_sched_config* cfg, int32_t n_requests, const int32_t* prompt_lens,
                                    const int32_t* response_lens, const int64_t* emit_offsets,
                                    const int32_t* emits, s3r_sched** out);

/*
 * Run one step.  rec (optional) receives its record; ran_ids (optional,
 * `capacity` entries) the ids of the requests in the round, in admission
 * order, and *n_ran their count (which may exceed capacity: then only the
 * first `capacity` ids are written).  *finished is set to 1 once every
 * request is done or the scheduler stalled; a step after that does nothing.
 */
S3R_API s3r_status s3r_sched_step(s3r_sched* s, s3r_sched_step_record* rec, int32_t* ran_ids, int32_t capacity,
                                  int32_t* n_ran, int32_t* finished);

/* Totals so far. */
S3R_API s3r_status s3r_sched_get_totals(const s3r_sched* s, s3r_sched_totals* out);

/* Free the scheduler (NULL is ignored). */
S3R_API void s3r_sched_destroy(s3r_sched* s);

/*
 * Create, step to completion (at most max_steps steps), destroy.  trace
 * (optional, max_steps records) receives every step's record.
 */
S3R_API s3r_status s3r_sched_run(const s3r_sched_config* cfg, int32_t n_requests, const int32_t* prompt_lens,
                                 const int32_t* response_lens, const int64_t* emit_offsets, const int32_t* emits,
                                 int64_t max_steps, s3r_sched_step_record* trace, s3r_sched_totals* out);

#ifdef __cplusplus
}
#endif

#endif /* S3R_SCHED_H_ */

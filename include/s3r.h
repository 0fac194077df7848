/*
 * s3r.h - C ABI of the S³R paged decode-attention hot path (B300, sm_103a).
 *
 * S³R (self-sparse speculative rollouts) drafts tokens with sparse attention
 * over a selected part of the KV history, verifies the drafted block with full
 * attention over the complete history, keeps the output distributed as the
 * dense policy through exact speculative sampling, and chooses the next
 * draft's history from the verification attention scores.  Sources: the
 * abstract of arXiv 2610.13202 ("S³R: Fast and Faithful RL Rollouts via
 * Self-Sparse Speculative Decoding"); the wispaper.ai summary, sections
 * "S3R drafts sparsely and verifies densely" and "Dense verification still
 * pays the full KV-cache bill"; the rebasdaily.com article, section
 * "草稿可以稀疏，交卷必须完整"; the rit.work blog, section "Как разреженный
 * черновик сохраняет ответы плотной модели".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Memory: every pointer is DEVICE memory owned by the caller unless the
 *    argument says "host".  The library allocates nothing and keeps no state
 *    between calls; scratch space comes from the caller's workspace.
 *  - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and the call returns at once.  Results and device
 *    errors are visible after the stream is synchronised.
 *  - Errors: argument and shape problems are found on the host and returned
 *    as a status before anything is enqueued.  Problems that only the data
 *    reveal (a page id or length outside the block table, a draft token
 *    outside the vocabulary, a bounded wait that ran out) never fault: the
 *    kernels skip the offending item, finish, and set a bit in the
 *    workspace's error word, read with s3r_read_device_error().  Outputs of a
 *    call that set an error bit are unspecified but finite.
 *  - Workspace: one caller-allocated device buffer of at least the size that
 *    the *_workspace_size() queries return, 256-byte aligned.  Its first 256
 *    bytes hold the sticky error word; the attention calls also keep
 *    per-(sequence, KV head) arrival counters in it, and the samplers
 *    per-sequence ones, which every call leaves at zero.  Zero the whole buffer once with s3r_workspace_init() after
 *    allocation, and again after a call reported S3R_DEVERR_TIMEOUT.  Calls
 *    that share a workspace must be ordered (same stream or event-ordered).
 *  - KV cache layout: bf16 pools [num_phys_pages][num_kv_heads][16][128]
 *    (one page holds 16 tokens; head_dim 128), addressed through a block
 *    table [num_seqs][max_pages_per_seq] of int32 physical page ids.  Query
 *    head qh reads KV head qh / (num_q_heads / num_kv_heads).
 *  - Precision: K, V and queries are bf16; scores, softmax and the weighted
 *    sum run in fp32 (the probabilities enter the bf16 tensor-core product as
 *    a bf16 high part plus a bf16 remainder); attention outputs are fp32.
 *  - Alignment: pools, queries and outputs 16-byte aligned.
 */
#ifndef S3R_H
#define S3R_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define S3R_API __attribute__((visibility("default")))
#else
#define S3R_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum s3r_status {
  S3R_OK = 0,
  S3R_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, inconsistent shapes */
  S3R_ERR_UNSUPPORTED = 2,  /* valid request outside what the kernels implement */
  S3R_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  S3R_ERR_WORKSPACE = 4     /* workspace missing, misaligned or too small */
} s3r_status;

/* Bits of the device error word (s3r_read_device_error). */
#define S3R_DEVERR_BAD_PAGE 0x1    /* block-table or selected page id out of range */
#define S3R_DEVERR_BAD_LENGTH 0x2  /* a length exceeds the block table (or is negative) */
#define S3R_DEVERR_BAD_TOKEN 0x4   /* a draft token outside [0, vocab) */
#define S3R_DEVERR_TIMEOUT 0x8     /* a bounded wait on a copy ran out */
#define S3R_DEVERR_BAD_COUNT 0x10  /* a selection count outside [0, b_max] */

#define S3R_PAGE_SIZE 16
#define S3R_HEAD_DIM 128
/* q rows that share one KV head in one call: (verify rows) x (q heads per KV head). */
#define S3R_MAX_ROWS_PER_KV_HEAD 32

/* The paged KV cache of one attention layer (all pointers device memory). */
typedef struct s3r_paged_kv {
  const void* k_pool;          /* bf16 [num_phys_pages][num_kv_heads][16][128] */
  const void* v_pool;          /* bf16, same layout as k_pool */
  int64_t num_phys_pages;
  const int32_t* block_table;  /* [num_seqs][max_pages_per_seq] physical page ids */
  int32_t max_pages_per_seq;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;            /* must be 128 */
  int32_t page_size;           /* must be 16 */
} s3r_paged_kv;

/* Library version string (host). */
S3R_API const char* s3r_version(void);

/* Human-readable name of a status (host). */
S3R_API const char* s3r_status_string(s3r_status status);

/*
 * Workspace bytes for the attention calls on `kv` with at most
 * `max_block_rows` verify rows (1 when only decode / draft calls are made),
 * on the current CUDA device (host).  Writes the size to *bytes.
 */
S3R_API s3r_status s3r_attn_workspace_size(const s3r_paged_kv* kv, int32_t max_block_rows, size_t* bytes);

/* Workspace bytes for s3r_spec_sample with n sequences and k drafts (host). */
S3R_API s3r_status s3r_spec_sample_workspace_size(int32_t n, int32_t k, size_t* bytes);

/* Workspace bytes for s3r_select_draft_pages (host): the error word only. */
S3R_API s3r_status s3r_select_workspace_size(size_t* bytes);

/* Zero the whole workspace: error word and counters (enqueued on `stream`). */
S3R_API s3r_status s3r_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronise `stream`, then copy the workspace's error word into *code
 * (host int).  If clear != 0 the word is reset to zero afterwards.
 */
S3R_API s3r_status s3r_read_device_error(const void* ws, void* stream, int32_t* code, int32_t clear);

/*
 * Dense autoregressive decode attention: the baseline S³R's speedups are
 * measured against (arXiv abstract: attention is 72-76% of autoregressive
 * decoding kernel time; wispaper.ai, "Sparse sampling changes the group, not
 * just the speed": each decoding step reads the KV cache of the whole
 * context).
 *
 *   q        bf16 [num_seqs][num_q_heads][128], the query of each sequence
 *   ctx_lens int32 [num_seqs]; the query attends to tokens 0..ctx_lens[s]-1
 *            (the count includes the current token, whose K/V are already
 *            in the pages); 0 gives a zero output row
 *   out      fp32 [num_seqs][num_q_heads][128]
 *   out[s][qh] = softmax(sm_scale * q[s][qh] . K_t) weighted sum of V_t.
 */
S3R_API s3r_status s3r_dense_decode_attn(const s3r_paged_kv* kv, const int32_t* ctx_lens, const void* q,
                                 void* out, float sm_scale, void* ws, size_t ws_bytes,
                                 void* stream);

/*
 * Budgeted sparse draft attention for draft step `draft_pos` (j >= 0): the
 * drafter is the policy itself reading only a selected part of the history
 * (wispaper.ai, "S3R drafts sparsely and verifies densely"; rebasdaily.com,
 * "草稿可以稀疏，交卷必须完整").
 *
 *   hist_lens int32 [num_seqs], L = history length before the draft block
 *   sel_pages int32 [num_seqs][num_kv_heads][b_max] distinct logical page
 *             ids in any order; the first sel_count entries are used
 *   sel_count int32 [num_seqs][num_kv_heads], each in [0, b_max]
 *   q         bf16 [num_seqs][num_q_heads][128]
 *   out       fp32 [num_seqs][num_q_heads][128]
 * Query head qh of sequence s attends to the tokens t < L whose page t/16 is
 * among the selected pages of its KV head, plus the draft tail L..L+j (their
 * K/V must already be in the pages).
 */
S3R_API s3r_status s3r_sparse_draft_attn(const s3r_paged_kv* kv, const int32_t* hist_lens,
                                 int32_t draft_pos, const int32_t* sel_pages,
                                 const int32_t* sel_count, int32_t b_max, const void* q, void* out,
                                 float sm_scale, void* ws, size_t ws_bytes, void* stream);

/*
 * Dense causal verification of a block of n_rows drafted positions against the
 * complete history (wispaper.ai, "S3R drafts sparsely and verifies densely":
 * full-attention verification in parallel; "Dense verification still pays
 * the full KV-cache bill").
 *
 *   hist_lens int32 [num_seqs], L
 *   q         bf16 [num_seqs][n_rows][num_q_heads][128]; row i is the query
 *             at position L+i and attends to tokens 0..L+i
 *   out       fp32 [num_seqs][n_rows][num_q_heads][128]
 *   page_mass optional (NULL to skip) fp32 [num_seqs][num_kv_heads][mass_stride]:
 *             for page pg < ceil((L+n_rows)/16), the sum over the KV head's
 *             query heads, the n_rows rows and the page's tokens of each row's
 *             normalised attention weight (each row contributes 1); entries
 *             from ceil((L+n_rows)/16) to mass_stride-1 are written as 0.
 *             mass_stride >= max_pages_per_seq.  This is the signal the
 *             next draft's history is chosen from (rit.work, "Как разреженный
 *             черновик сохраняет ответы плотной модели").
 * Requires n_rows * (num_q_heads / num_kv_heads) <= S3R_MAX_ROWS_PER_KV_HEAD.
 */
S3R_API s3r_status s3r_verify_attn(const s3r_paged_kv* kv, const int32_t* hist_lens, int32_t n_rows,
                           const void* q, void* out, float* page_mass, int32_t mass_stride,
                           float sm_scale, void* ws, size_t ws_bytes, void* stream);

/*
 * The three attention calls above with their new K/V rows written into the
 * pages in the same launch, before they are read: the drafter's row of the
 * current token, and verification's dense rows of the block (wispaper.ai, "S3R
 * drafts sparsely and verifies densely": the accepted part of the block keeps
 * its dense states).  Each equals s3r_kv_append of those rows followed by the
 * plain call, in results and in the pages it leaves, without the separate
 * launch.
 *
 *   rows.k_rows, rows.v_rows  bf16 [num_seqs][rows.n_rows][num_kv_heads][128],
 *                16-byte aligned
 *   dense decode: n_rows = 1, the row of position ctx_lens[s] - 1 (none for a
 *                 sequence with ctx_lens[s] = 0: it reads nothing and writes
 *                 nothing, and its output rows are zero)
 *   sparse draft: n_rows = 1, the row of position hist_lens[s] + draft_pos
 *   verify:       n_rows = the call's n_rows, rows of positions
 *                 hist_lens[s] .. hist_lens[s] + n_rows - 1
 * A row whose page id is outside the pool is not written (and that page is not
 * read: the call reports S3R_DEVERR_BAD_PAGE).  The pages that receive rows
 * must not be shared with another sequence of the call.  The pool descriptor's
 * k_pool and v_pool are written; the rows are caller-owned device memory, read
 * only.  A missing rows struct returns S3R_ERR_INVALID_ARG at once; after the
 * plain call's own checks, so do rows.n_rows other than stated above and a
 * null or unaligned row pointer.  Nothing is enqueued in either case.
 */
typedef struct s3r_kv_rows {
  const void* k_rows;
  const void* v_rows;
  int32_t n_rows;
} s3r_kv_rows;

S3R_API s3r_status s3r_dense_decode_attn_append(const s3r_paged_kv* kv, const int32_t* ctx_lens,
                                        const s3r_kv_rows* rows, const void* q, void* out, float sm_scale,
                                        void* ws, size_t ws_bytes, void* stream);

S3R_API s3r_status s3r_sparse_draft_attn_append(const s3r_paged_kv* kv, const int32_t* hist_lens,
                                        int32_t draft_pos, const int32_t* sel_pages,
                                        const int32_t* sel_count, int32_t b_max, const s3r_kv_rows* rows,
                                        const void* q, void* out, float sm_scale, void* ws, size_t ws_bytes,
                                        void* stream);

S3R_API s3r_status s3r_verify_attn_append(const s3r_paged_kv* kv, const int32_t* hist_lens, int32_t n_rows,
                                  const s3r_kv_rows* rows, const void* q, void* out, float* page_mass,
                                  int32_t mass_stride, float sm_scale, void* ws, size_t ws_bytes,
                                  void* stream);

/*
 * Choose the next draft's KV pages per (sequence, KV head) from the verify
 * page mass.  The pages say the attention scores choose the history (rit.work,
 * same section) and that selection must stay cheap (wispaper.ai, "Where the
 * speedup claim holds"); the rule is this library's:
 *   P = ceil(sel_lens[s] / 16); M = pages [0, n_sink) and [P - n_recent, P)
 *   B = min(P, max(ceil(budget * P - 1e-9), |M|))   (fp64 arithmetic)
 *   B == P: all pages; else M plus the B - |M| other pages of largest mass,
 *   equal mass -> lower page id first.
 *
 *   page_mass fp32 [num_seqs][num_kv_heads][mass_stride]
 *   sel_lens  int32 [num_seqs]; requires ceil(sel_lens/16) <= mass_stride
 *   sel_pages int32 [num_seqs][num_kv_heads][b_max] out: ascending page ids,
 *             unused slots set to -1
 *   sel_count int32 [num_seqs][num_kv_heads] out: B
 * b_max must be at least the B of a history of mass_stride pages;
 * mass_stride above 49152 pages returns S3R_ERR_UNSUPPORTED.
 */
S3R_API s3r_status s3r_select_draft_pages(const float* page_mass, const int32_t* sel_lens, int32_t num_seqs,
                                  int32_t num_kv_heads, int32_t mass_stride, double budget,
                                  int32_t n_sink, int32_t n_recent, int32_t* sel_pages,
                                  int32_t* sel_count, int32_t b_max, void* ws, size_t ws_bytes,
                                  void* stream);

/*
 * Exact speculative sampling of n drafted blocks of k tokens (wispaper.ai,
 * "S3R drafts sparsely and verifies densely": exact speculative sampling
 * preserves the target distribution; rebasdaily.com and rit.work: a rejected
 * draft is replaced by a token from the corrected / residual distribution).
 *
 *   p_logits     fp32 [n][k+1][vocab] target logits for block positions 1..k+1
 *   q_logits     fp32 [n][k][vocab]   draft logits for positions 1..k
 *   draft_tokens int32 [n][k]
 *   out_tokens   int32 [n][k+1] out: accepted drafts, then the correcting or
 *                bonus token, then -1
 *   n_accepted   int32 [n] out
 *   tie_count    optional (NULL to skip) uint32 [2] out, zeroed by the call:
 *                [0] the ratio tests, up to and including each sequence's
 *                first rejection, whose uniform lies within 1e-6 of the
 *                ratio (|u - p_i(x_i)/q_i(x_i)| <= 1e-6); [1] the sequences
 *                whose inverse-CDF target u*Z lies within 1e-6*Z of either end
 *                of the picked token's interval of the running sum (or that
 *                took the rounding fallback).  These are the decisions that
 *                rounding in the fp32 row statistics could flip against an
 *                exact evaluation; the tokens stay valid samples, and the
 *                counts say how many such decisions a call made.
 * With p_i = softmax(p_logits[i]), q_i = softmax(q_logits[i]) (temperature 1),
 * draft x_i is accepted iff u < p_i(x_i) / q_i(x_i), u = Philox4x32-10 uniform
 * of counter (n, i-1, 0, offset) and key seed; at the first rejection the
 * token is the inverse CDF (token-id order) of max(0, p_i - q_i) at the
 * uniform of counter (n, i-1, 1, offset); if all k are accepted the bonus
 * token is the inverse CDF of p_{k+1} at counter (n, k, 1, offset).  A
 * uniform is (first output word >> 8) * 2^-24.  offset must be < 2^32.
 */
S3R_API s3r_status s3r_spec_sample(const float* p_logits, const float* q_logits,
                           const int32_t* draft_tokens, int32_t n, int32_t k, int32_t vocab,
                           uint64_t seed, uint64_t offset, int32_t* out_tokens,
                           int32_t* n_accepted, uint32_t* tie_count, void* ws, size_t ws_bytes,
                           void* stream);

/*
 * Exact speculative sampling with the ratio tests taken one draft position at
 * a time: the rows of a sequence after its first rejection (p_j and q_j for
 * j > a) are never read, and the bonus row p_{k+1} only when all k drafts
 * were accepted.  The drafts are tested in order and sampling stops at the
 * first rejection (wispaper.ai, "S3R drafts sparsely and verifies densely";
 * rebasdaily.com, "草稿可以稀疏，交卷必须完整"), so the skipped rows cannot
 * change the result.
 *
 * Same arguments, semantics, results (bit for bit, tie counts included) and
 * workspace size as s3r_spec_sample.  It enqueues k + 3 kernels instead of one
 * (plus a clear of tie_count when given) and reads about
 * (2 E[a] + 2) / (2k + 1) of the logit bytes, E[a] the mean accepted count.
 * Its workspace must hold zeroed arrival counters (s3r_workspace_init once
 * after allocation); every call leaves them at zero.
 */
S3R_API s3r_status s3r_spec_sample_sequential(const float* p_logits, const float* q_logits,
                                      const int32_t* draft_tokens, int32_t n, int32_t k, int32_t vocab,
                                      uint64_t seed, uint64_t offset, int32_t* out_tokens,
                                      int32_t* n_accepted, uint32_t* tie_count, void* ws, size_t ws_bytes,
                                      void* stream);

/* Workspace bytes for s3r_sample_draft_tokens with n sequences (host). */
S3R_API s3r_status s3r_sample_draft_workspace_size(int32_t n, size_t* bytes);

/*
 * Draft-token sampling: the drafter proposes each token by sampling from its
 * own distribution q (wispaper.ai, "S3R drafts sparsely and verifies densely";
 * rebasdaily.com, "草稿可以稀疏，交卷必须完整"), here at draft step
 * `draft_pos` of every sequence.
 *
 *   logits        fp32, row s (vocab values) at logits + s * row_stride; the
 *                 drafter's logits at this step.  row_stride >= vocab
 *                 (elements), so the rows may be one slice [n][j][vocab] of
 *                 a [n][k][vocab] block of draft logits (row_stride = k*vocab)
 *   tokens        int32 out: token s at tokens[s * token_stride]
 *                 (token_stride >= 1, e.g. k for column j of [n][k] drafts)
 * token[s] is the inverse CDF, in token-id order, of softmax(logits[s])
 * (temperature 1) at the Philox4x32-10 uniform of counter
 * (s, draft_pos, 2, offset) and key seed (stream 2 = DRAFT), with the same
 * uniform and inverse-CDF conventions as s3r_spec_sample.  offset < 2^32.
 * Its workspace must hold zeroed arrival counters (s3r_workspace_init once);
 * every call leaves them at zero.
 */
S3R_API s3r_status s3r_sample_draft_tokens(const float* logits, int32_t n, int32_t vocab, int64_t row_stride,
                                   uint64_t seed, uint64_t offset, int32_t draft_pos, int32_t* tokens,
                                   int64_t token_stride, void* ws, size_t ws_bytes, void* stream);

/*
 * Append a block of K/V rows to every sequence's paged cache.  The drafter
 * writes the row of each draft step, and verification the dense rows of the
 * verified block, which the system keeps for the accepted part (wispaper.ai,
 * "S3R drafts sparsely and verifies densely"; rit.work, "Как разреженный
 * черновик сохраняет ответы плотной модели").
 *
 *   kv          the layer's cache; its k_pool and v_pool are WRITTEN (they
 *               are const in s3r_paged_kv because attention only reads them)
 *   start_lens  int32 [num_seqs]: position of row 0 (the length L before it)
 *   n_rows      int32 [num_seqs] rows to write per sequence, in [0, max_rows];
 *               NULL writes max_rows rows for every sequence
 *   k_rows, v_rows  bf16 [num_seqs][max_rows][num_kv_heads][128], 16-byte
 *               aligned; row t of sequence s goes to position L + t: slot
 *               (L + t) % 16 of page block_table[s][(L + t) / 16]
 * Rows beyond the block table set S3R_DEVERR_BAD_LENGTH, page ids outside the
 * pool S3R_DEVERR_BAD_PAGE, and a count outside [0, max_rows]
 * S3R_DEVERR_BAD_COUNT; such rows are not written.  ws: any workspace of at
 * least 256 bytes (its error word is used).
 */
S3R_API s3r_status s3r_kv_append(const s3r_paged_kv* kv, const int32_t* start_lens, const int32_t* n_rows,
                                 int32_t max_rows, const void* k_rows, const void* v_rows, void* ws,
                                 size_t ws_bytes, void* stream);

/*
 * Commit a verified block: new_lens[s] = hist_lens[s] + n_accepted[s] + 1,
 * the pending token and the accepted drafts, whose dense rows the block's
 * s3r_kv_append wrote at positions L .. L + n_accepted.  The rejected drafts'
 * rows lie past the new length: they are dropped (rolled back) and the next
 * round's appends overwrite them (rebasdaily.com and rit.work: a rejected
 * draft and everything after it is discarded).
 *
 *   hist_lens, n_accepted  int32 [n]; new_lens int32 [n] out (may be hist_lens)
 * n_accepted outside [0, max_accept] sets S3R_DEVERR_BAD_COUNT and a new length
 * above max_len S3R_DEVERR_BAD_LENGTH; such a sequence keeps its length.
 * ws: any workspace of at least 256 bytes.
 */
S3R_API s3r_status s3r_commit_lengths(const int32_t* hist_lens, const int32_t* n_accepted, int32_t n,
                                      int32_t max_accept, int32_t max_len, int32_t* new_lens, void* ws,
                                      size_t ws_bytes, void* stream);

/* Bytes of library-owned device scratch behind s3r_spec_sample_noalloc, held
 * once by every GPU that loads the library until the process exits. */
#define S3R_NOALLOC_SCRATCH_BYTES (2u * 1024u * 1024u)

/*
 * s3r_spec_sample for callers that cannot allocate device memory: code whose
 * device memory is one pool reserved up front, plugins that are handed only
 * their input and output buffers, runtimes that forbid cudaMalloc once they
 * are serving.  The S³R pages have no counterpart to this call; it exists
 * only for such callers.
 *
 * Same arguments, semantics and results as s3r_spec_sample, without
 * tie_count, ws and ws_bytes.  Its scratch is a fixed
 * S3R_NOALLOC_SCRATCH_BYTES array in the library's device image, so it never
 * calls cudaMalloc, cudaFree or any allocating routine.
 *   device_error  optional (NULL to skip) device int32 that receives this
 *                 call's device error bits (the S3R_DEVERR_* values)
 * Returns S3R_ERR_UNSUPPORTED, before enqueuing anything, when
 * s3r_spec_sample_workspace_size(n, k) exceeds S3R_NOALLOC_SCRATCH_BYTES
 * (for example n = 2048 with k = 8 needs 1,884,672 bytes and fits).  Every
 * other argument error also returns before anything is enqueued.
 * The stream and every pointer must belong to the CURRENT device: the call
 * uses the current device's copy of the array.  The first call on each
 * device looks up the array's device address (a one-time set-up per device,
 * with that device current): make that first call before any stream capture.
 * A call that fails with S3R_ERR_CUDA drops the cached address, and the next
 * call looks it up again; a device reset (cudaDeviceReset) between calls is
 * not otherwise supported.  Every call on a device shares the one array and
 * overwrites it, so calls whose work may overlap on the GPU (different
 * streams without ordering) race and must not be issued.
 */
S3R_API s3r_status s3r_spec_sample_noalloc(const float* p_logits, const float* q_logits,
                                   const int32_t* draft_tokens, int32_t n, int32_t k, int32_t vocab,
                                   uint64_t seed, uint64_t offset, int32_t* out_tokens,
                                   int32_t* n_accepted, int32_t* device_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* S3R_H */

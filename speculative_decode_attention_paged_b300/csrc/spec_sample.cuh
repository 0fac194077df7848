// Exact speculative sampler: workspace layout and host launch interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/s3r.h"

namespace s3r {

// Largest draft length the samplers take.
constexpr int kMaxSpecK = 64;

// Each residual (or bonus) row is cut into this many contiguous chunks; the
// chunk sums locate the inverse-CDF target before one chunk is scanned.
constexpr int kSampleChunks = 32;

struct SpecWorkspaceLayout {
  size_t err_off;     // device error word (first 256 bytes)
  size_t stats_off;   // float2 [N][2k+1]: (row max, sum of exp(x - max))
  size_t accept_off;  // int32 [N]: accepted count a = index of the row sampled from
  size_t chunk_off;   // double2 [N][kSampleChunks]: (residual sum, target-row sum) per chunk
  size_t bonus_off;   // float2 [N][kSampleChunks]: (max, sum) per chunk of the bonus row p_k
  size_t arrive_off;      // int32 [N]: per-sequence arrival counters, zero between calls
  size_t res_arrive_off;  // int32 [N]: per-sequence chunk-sum arrivals, zero between calls
  size_t ready_off;       // int32 [N]: per-sequence "ratio tests done" flags, zero between calls
  size_t ticket_off;      // int32 [2]: task ticket and finished-CTA count, zero between calls
  size_t total;           // the counters [arrive_off, total) are contiguous
};

SpecWorkspaceLayout spec_workspace_layout(int64_t N, int k);

// Host checks of the sampler's arguments other than the workspace (sizes,
// offset, null pointers); S3R_OK or the status to return before enqueuing.
s3r_status check_spec_sample_args(const float* p_logits, const float* q_logits, const int32_t* draft_tokens,
                                  int32_t n, int32_t k, int32_t vocab, uint64_t offset, const int32_t* out_tokens,
                                  const int32_t* n_accepted);

// Enqueue the sampler kernels.  `ws` is the caller's workspace laid out by
// spec_workspace_layout(N, k).  With k > 0 the final inverse CDF draws the
// Philox uniform of counter (n, a, RESAMPLE, offset), a the accepted count.
// With k = 0 (no draft rows) one token is sampled from softmax(p) per sequence
// with the uniform of counter (n, u_pos, u_stream, offset), u_pos < 0 meaning
// 0, and n_accepted is set to 0; then row n is read at p + n * row_stride
// (0: V) and its token written to out_tokens[n * token_stride].
// ties (nullable, two counters the caller has zeroed): [0] gains the ratio
// tests with |u - p/q| <= 1e-6 up to each sequence's first rejection, [1] the
// inverse-CDF picks whose target lies within 1e-6 * Z of an end of the picked
// token's interval.
cudaError_t launch_spec_sample(const float* p, const float* q, const int32_t* drafts, int N, int k,
                               int V, uint64_t seed, uint32_t offset, void* ws,
                               int32_t* out_tokens, int32_t* n_accepted, cudaStream_t stream,
                               uint32_t u_stream = 1, int u_pos = -1, int64_t row_stride = 0,
                               int64_t token_stride = 1, uint32_t* ties = nullptr);

// The same sampling with the ratio tests taken one position at a time
// (k + 1 step launches): a sequence's rows after its first rejection are
// never read.  Same outputs as launch_spec_sample.
cudaError_t launch_spec_sample_sequential(const float* p, const float* q, const int32_t* drafts, int N, int k,
                                          int V, uint64_t seed, uint32_t offset, void* ws,
                                          int32_t* out_tokens, int32_t* n_accepted, cudaStream_t stream,
                                          uint32_t* ties = nullptr);

}  // namespace s3r

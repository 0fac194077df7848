// Paged split-KV attention engine shared by the three attention forms of an
// S³R round: dense decode, budgeted sparse draft, dense causal verify (+ page
// mass).  Host-visible launch interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace s3r {

enum AttnMode : int { kModeDense = 0, kModeSparse = 1, kModeVerify = 2 };

constexpr int kAttnWarps = 8;       // warps per CTA, each an independent worker
// TMA stages per warp (one (page, KV head) K+V tile each): two stages (128 KiB
// in flight per SM) stream faster than three (192 KiB), which only queue
// longer in DRAM.
constexpr int kAttnStages = 2;
constexpr int kPairChunk = 32;      // (sequence, KV head) pairs per prefix-sum chunk
constexpr int kMaxPairs = 262144;   // chunk prefix must fit in shared memory

struct AttnArgs {
  int mode;
  int S, Hq, Hkv, G, T, R;          // R = T * G query rows per (sequence, KV head) pair
  int max_pages;
  int64_t num_phys_pages;
  const int32_t* block_table;
  const int32_t* lens;              // ctx_lens (dense) or hist_lens (sparse, verify)
  int draft_pos;
  const int32_t* sel_pages;
  const int32_t* sel_count;
  int b_max;
  const __nv_bfloat16* q;
  float* out;                       // fp32 attention output
  float scale_log2;                 // sm_scale * log2(e)
  float* page_mass;                 // verify only, may be null
  int mass_stride;
  // K/V rows written into the pages before they are read (app_rows == 0: none):
  // bf16 [S][app_rows][Hkv][128], as 16-byte pieces; the first at position
  // ctx_len - 1 (dense), hist_len + draft_pos (sparse) or hist_len (verify)
  const uint4* app_k;
  const uint4* app_v;
  int app_rows;
  uint4* k_pool_w;                  // the pools the tensor maps read, for those writes
  uint4* v_pool_w;
  // workspace views
  int* err;
  int* arrivals;                    // [n_pairs] segments of a cut pair published so far
  float* part_o;                    // [2 * total_warps][R][128]
  float* part_ml;                   // [2 * total_warps][R][2]
  float* page_lse;                  // [n_pairs][max_pages][R]  (page mass only)
  int total_warps;
  int n_pairs;
  int n_chunks;
  // Test of the bounded waits only (0 otherwise): the tcgen05 verify kernel's CTA 0
  // loads no K for its first tile and never arrives on that tile's barrier, so the
  // waits on it run out and the abort path runs (see s3r_test_stall_next_verify).
  int test_stall;
};

struct AttnWorkspaceLayout {
  size_t err_off, arrivals_off, part_o_off, part_ml_off, page_lse_off, total;
};

// Byte layout of the attention workspace for the given geometry.
AttnWorkspaceLayout attn_workspace_layout(int n_pairs, int rows, int max_pages, int total_warps,
                                          bool with_mass);

size_t attn_smem_bytes(int n_chunks);

// Enqueue the attention kernel.  `a` must be fully populated; the workspace's
// arrival counters must be zero (every call leaves them zero).
cudaError_t launch_attention(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a,
                             int grid, cudaStream_t stream);

// Verify on tcgen05 (rows per KV head <= 32): dynamic shared memory it needs
// for `n_chunks` chunks of 32 pairs, and the launch (qmap: 4-D view of the
// queries [S][T][Hq][128], box (64, G, T, 1), 128-byte swizzle).
size_t verify_tc_smem_bytes(int n_chunks);
cudaError_t launch_verify_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                             const AttnArgs& a, int grid, cudaStream_t stream);

}  // namespace s3r

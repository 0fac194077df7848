// KV append and length commit: host launch interface.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace s3r {

struct KvAppendArgs {
  void* k_pool;                 // bf16 [num_phys_pages][Hkv][16][128]
  void* v_pool;
  const int32_t* block_table;   // [S][max_pages]
  int64_t num_phys_pages;
  int max_pages;
  int S, Hkv;
  const int32_t* start_lens;    // [S]
  const int32_t* n_rows;        // [S] or null (all max_rows)
  int max_rows;
  const void* k_rows;           // bf16 [S][max_rows][Hkv][128]
  const void* v_rows;
  int* err;
};

cudaError_t launch_kv_append(const KvAppendArgs& a, cudaStream_t stream);

cudaError_t launch_commit_lengths(const int32_t* hist_lens, const int32_t* n_accepted, int n, int max_accept,
                                  int max_len, int32_t* new_lens, int* err, cudaStream_t stream);

}  // namespace s3r

// KV append and length commit for a closed S³R round.
//
// The S³R pages: the drafter reads a selected part of the history and
// proposes a block; verification runs the dense policy over the block and
// keeps the accepted prefix, whose dense states the system recomputes for the
// cache (wispaper.ai, "S3R drafts sparsely and verifies densely"; rit.work,
// "Как разреженный черновик сохраняет ответы плотной модели").  In a paged
// cache that is two operations:
//   kv_append   write a block of K/V rows (a draft step's row, or the dense
//               rows of the verified block) at positions L, L+1, ... of each
//               sequence, through its block table;
//   commit      advance each length by the accepted count plus the pending
//               token, L + n_acc + 1.  Rows past the new length (the rejected
//               drafts) are no longer part of the sequence and are overwritten
//               by the next round's appends: that is the rollback.

#include "kv_append.cuh"
#include "s3r_device.cuh"

namespace s3r {

namespace {

constexpr int kAppendWarps = 8;
constexpr int kRowVec = kHeadDim * 2 / 16;   // 16-byte pieces in one 128-wide bf16 row

// One warp per (sequence, block row): the row's K and V vectors of every KV
// head (2 x Hkv x 256 bytes) are copied with 16-byte loads and stores into
// slot (L + t) % 16 of page block_table[s][(L + t) / 16].
__global__ void __launch_bounds__(kAppendWarps * 32) kv_append_kernel(KvAppendArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t item = static_cast<int64_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
  if (item >= static_cast<int64_t>(a.S) * a.max_rows) return;
  const int s = static_cast<int>(item / a.max_rows);
  const int t = static_cast<int>(item - static_cast<int64_t>(s) * a.max_rows);
  const int n = a.n_rows != nullptr ? __ldg(a.n_rows + s) : a.max_rows;
  if (n < 0 || n > a.max_rows) {
    if (t == 0 && lane == 0) report_error(a.err, S3R_DEVERR_BAD_COUNT);
    return;
  }
  if (t >= n) return;
  const int L = __ldg(a.start_lens + s);
  const int64_t pos = static_cast<int64_t>(L) + t;
  if (L < 0 || pos >= static_cast<int64_t>(a.max_pages) * kPage) {
    if (lane == 0) report_error(a.err, S3R_DEVERR_BAD_LENGTH);
    return;
  }
  const int page = __ldg(a.block_table + static_cast<int64_t>(s) * a.max_pages + pos / kPage);
  if (page < 0 || page >= a.num_phys_pages) {
    if (lane == 0) report_error(a.err, S3R_DEVERR_BAD_PAGE);
    return;
  }
  const int slot = static_cast<int>(pos % kPage);
  const int per_row = 2 * a.Hkv * kRowVec;   // K pieces then V pieces
  for (int i = lane; i < per_row; i += 32) {
    const int is_v = i >= a.Hkv * kRowVec;
    const int j = is_v ? i - a.Hkv * kRowVec : i;
    const int h = j / kRowVec, piece = j - h * kRowVec;
    const uint4* src = reinterpret_cast<const uint4*>(is_v ? a.v_rows : a.k_rows) +
                       ((item * a.Hkv + h) * kRowVec + piece);
    uint4* dst = reinterpret_cast<uint4*>(is_v ? a.v_pool : a.k_pool) +
                 (((static_cast<int64_t>(page) * a.Hkv + h) * kPage + slot) * kRowVec + piece);
    *dst = __ldg(src);
  }
}

// One thread per sequence: L + n_acc + 1, or L unchanged (and an error bit)
// when n_acc is outside [0, max_accept] or the new length exceeds max_len.
__global__ void commit_lengths_kernel(const int32_t* hist_lens,
                                      const int32_t* __restrict__ n_accepted, int n, int max_accept,
                                      int max_len, int32_t* new_lens, int* err) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n) return;
  const int L = hist_lens[s];
  const int a = n_accepted[s];
  int out = L;
  if (a < 0 || a > max_accept) {
    report_error(err, S3R_DEVERR_BAD_COUNT);
  } else if (L < 0 || static_cast<int64_t>(L) + a + 1 > max_len) {
    report_error(err, S3R_DEVERR_BAD_LENGTH);
  } else {
    out = L + a + 1;
  }
  new_lens[s] = out;
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendArgs& a, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(a.S) * a.max_rows;
  if (items == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((items + kAppendWarps - 1) / kAppendWarps);
  kv_append_kernel<<<blocks, kAppendWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_commit_lengths(const int32_t* hist_lens, const int32_t* n_accepted, int n, int max_accept,
                                  int max_len, int32_t* new_lens, int* err, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  commit_lengths_kernel<<<(n + 255) / 256, 256, 0, stream>>>(hist_lens, n_accepted, n, max_accept, max_len,
                                                             new_lens, err);
  return cudaGetLastError();
}

}  // namespace s3r

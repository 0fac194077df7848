// C ABI of the S³R hot path: host-side validation, workspace layout, TMA
// descriptors and kernel launches.  Declarations and contracts: include/s3r.h.

#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "attn_paged.cuh"
#include "s3r_device.cuh"
#include "spec_sample.cuh"
#include "kv_append.cuh"
#include "../../include/s3r_testing.h"

namespace s3r {

s3r_status check_spec_sample_args(const float* p_logits, const float* q_logits, const int32_t* draft_tokens,
                                  int32_t n, int32_t k, int32_t vocab, uint64_t offset, const int32_t* out_tokens,
                                  const int32_t* n_accepted) {
  if (n < 0 || k < 0 || vocab <= 0) return S3R_ERR_INVALID_ARG;
  if (k > kMaxSpecK) return S3R_ERR_UNSUPPORTED;
  if (offset > 0xffffffffULL) return S3R_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n) * (k + 1) * vocab > (int64_t{1} << 40)) return S3R_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(n) * std::max(2 * k + 1, kSampleChunks) > 0x7fffffffLL) return S3R_ERR_UNSUPPORTED;
  if (n == 0) return S3R_OK;
  if (p_logits == nullptr || out_tokens == nullptr || n_accepted == nullptr) return S3R_ERR_INVALID_ARG;
  if (k > 0 && (q_logits == nullptr || draft_tokens == nullptr)) return S3R_ERR_INVALID_ARG;
  return S3R_OK;
}

cudaError_t launch_select_pages(const float* mass, const int32_t* sel_lens, int S, int Hkv,
                                int stride, double budget, int n_sink, int n_recent,
                                int32_t* sel_pages, int32_t* sel_count, int b_max, int* err,
                                cudaStream_t stream);
}  // namespace s3r

namespace {

using namespace s3r;

constexpr int kMaxDevices = 64;
constexpr uint32_t kStreamDraftU = 2;   // Philox stream of draft-token sampling
// Longest mass row the selection kernel stages in shared memory (pages).
constexpr int kMaxSelectPages = 49152;

int g_sm_count[kMaxDevices];
std::once_flag g_encode_once;
// s3r_test_stall_next_verify: armed for the next tcgen05 verify launch only.
std::atomic<int> g_test_stall{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// SM count of the current device (cached), or 0 on failure.
int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  });
  return g_encode;
}

// 3-D view of a KV pool: (d: 128, row: kv_heads*16, page: num_phys_pages);
// box (64, 16, 1) = one 64-column half of a (page, KV head) tile, 128B swizzle.
bool encode_pool_map(CUtensorMap* map, const void* pool, int kv_heads, int64_t num_pages) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(kv_heads) * kPage,
                        static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                           static_cast<cuuint64_t>(kv_heads) * kPage * kHeadDim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kPage), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D view of the verify queries q [S][T][Hq][128] bf16: box (64, G, T, 1)
// = one 64-column half of the T x G query rows of one (sequence, KV head).
bool encode_query_map(CUtensorMap* map, const void* q, int S, int T, int Hq, int G) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(Hq),
                        static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(S)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                           static_cast<cuuint64_t>(Hq) * kHeadDim * 2,
                           static_cast<cuuint64_t>(T) * Hq * kHeadDim * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(T), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Largest dynamic shared memory a block may opt into on the current device.
size_t max_dynamic_smem() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  return static_cast<size_t>(v);
}

s3r_status validate_kv(const s3r_paged_kv* kv) {
  if (kv == nullptr) return S3R_ERR_INVALID_ARG;
  if (kv->head_dim != kHeadDim || kv->page_size != kPage) return S3R_ERR_UNSUPPORTED;
  if (kv->num_seqs < 0 || kv->num_kv_heads <= 0 || kv->num_q_heads <= 0 ||
      kv->max_pages_per_seq <= 0 || kv->num_phys_pages <= 0)
    return S3R_ERR_INVALID_ARG;
  if (kv->num_q_heads % kv->num_kv_heads != 0) return S3R_ERR_INVALID_ARG;
  if (kv->num_phys_pages > 0x7fffffffLL) return S3R_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(kv->max_pages_per_seq) * kPage > 0x3fffffff) return S3R_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(kv->num_seqs) * kv->num_kv_heads > kMaxPairs) return S3R_ERR_UNSUPPORTED;
  // the global page stream is indexed with 32-bit counts
  if (static_cast<int64_t>(kv->num_seqs) * kv->num_kv_heads * kv->max_pages_per_seq > 0x7fffffffLL)
    return S3R_ERR_UNSUPPORTED;
  if (kv->num_seqs > 0) {
    if (kv->k_pool == nullptr || kv->v_pool == nullptr || kv->block_table == nullptr)
      return S3R_ERR_INVALID_ARG;
    if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool)) return S3R_ERR_INVALID_ARG;
  }
  return S3R_OK;
}

s3r_status to_status(cudaError_t e) { return e == cudaSuccess ? S3R_OK : S3R_ERR_CUDA; }

// Shared body of the three attention calls.
s3r_status run_attention(const s3r_paged_kv* kv, int mode, const int32_t* lens, int T,
                         int draft_pos, const int32_t* sel_pages, const int32_t* sel_count,
                         int b_max, const void* q, void* out, float* page_mass, int mass_stride,
                         float sm_scale, void* ws, size_t ws_bytes, void* stream,
                         const s3r_kv_rows* rows = nullptr) {
  s3r_status st = validate_kv(kv);
  if (st != S3R_OK) return st;
  if (!std::isfinite(sm_scale)) return S3R_ERR_INVALID_ARG;
  const int G = kv->num_q_heads / kv->num_kv_heads;
  const int R = T * G;
  if (T <= 0) return S3R_ERR_INVALID_ARG;
  if (R > S3R_MAX_ROWS_PER_KV_HEAD) return S3R_ERR_UNSUPPORTED;
  if (ws == nullptr || !aligned256(ws)) return S3R_ERR_WORKSPACE;
  if (kv->num_seqs == 0) return S3R_OK;
  if (lens == nullptr || q == nullptr || out == nullptr) return S3R_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return S3R_ERR_INVALID_ARG;
  if (mode == kModeSparse) {
    if (draft_pos < 0 || b_max < 0 || (b_max > 0 && sel_pages == nullptr) || sel_count == nullptr)
      return S3R_ERR_INVALID_ARG;
  }
  const bool mass = page_mass != nullptr;
  if (mass && mass_stride < kv->max_pages_per_seq) return S3R_ERR_INVALID_ARG;
  if (rows != nullptr) {
    if (rows->n_rows != (mode == kModeVerify ? T : 1)) return S3R_ERR_INVALID_ARG;
    if (rows->k_rows == nullptr || rows->v_rows == nullptr) return S3R_ERR_INVALID_ARG;
    if (!aligned16(rows->k_rows) || !aligned16(rows->v_rows)) return S3R_ERR_INVALID_ARG;
  }

  const int sms = current_sm_count();
  if (sms <= 0) return S3R_ERR_CUDA;
  const int total_warps = sms * kAttnWarps;
  const int n_pairs = kv->num_seqs * kv->num_kv_heads;
  const AttnWorkspaceLayout lay =
      attn_workspace_layout(n_pairs, R, kv->max_pages_per_seq, total_warps, mass);
  if (ws_bytes < lay.total) return S3R_ERR_WORKSPACE;

  CUtensorMap kmap, vmap;
  if (!encode_pool_map(&kmap, kv->k_pool, kv->num_kv_heads, kv->num_phys_pages) ||
      !encode_pool_map(&vmap, kv->v_pool, kv->num_kv_heads, kv->num_phys_pages))
    return S3R_ERR_CUDA;

  uint8_t* w = static_cast<uint8_t*>(ws);
  AttnArgs a{};
  a.mode = mode;
  a.S = kv->num_seqs;
  a.Hq = kv->num_q_heads;
  a.Hkv = kv->num_kv_heads;
  a.G = G;
  a.T = T;
  a.R = R;
  a.max_pages = kv->max_pages_per_seq;
  a.num_phys_pages = kv->num_phys_pages;
  a.block_table = kv->block_table;
  a.lens = lens;
  a.draft_pos = draft_pos;
  a.sel_pages = sel_pages;
  a.sel_count = sel_count;
  a.b_max = b_max;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.out = static_cast<float*>(out);
  a.scale_log2 = sm_scale * kLog2e;
  a.page_mass = page_mass;
  a.mass_stride = mass_stride;
  a.err = reinterpret_cast<int*>(w + lay.err_off);
  a.arrivals = reinterpret_cast<int*>(w + lay.arrivals_off);
  a.part_o = reinterpret_cast<float*>(w + lay.part_o_off);
  a.part_ml = reinterpret_cast<float*>(w + lay.part_ml_off);
  a.page_lse = mass ? reinterpret_cast<float*>(w + lay.page_lse_off) : nullptr;
  if (rows != nullptr) {
    a.app_k = static_cast<const uint4*>(rows->k_rows);
    a.app_v = static_cast<const uint4*>(rows->v_rows);
    a.app_rows = rows->n_rows;
    // the pools are declared const in s3r_paged_kv because plain attention only reads them
    a.k_pool_w = static_cast<uint4*>(const_cast<void*>(kv->k_pool));
    a.v_pool_w = static_cast<uint4*>(const_cast<void*>(kv->v_pool));
  }
  a.total_warps = total_warps;
  a.n_pairs = n_pairs;
  a.n_chunks = (n_pairs + kPairChunk - 1) / kPairChunk;
  // Verify with more than 16 query rows per KV head runs on the tcgen05
  // kernel (the CUDA-core kernel would hold two 16-row MMA tiles per warp and
  // spill); up to 16 rows the CUDA-core kernel streams at the copy bandwidth.
  if (mode == kModeVerify && R > 16 && R <= S3R_MAX_ROWS_PER_KV_HEAD &&
      verify_tc_smem_bytes(a.n_chunks) <= max_dynamic_smem()) {
    CUtensorMap qmap;
    if (!encode_query_map(&qmap, q, kv->num_seqs, T, kv->num_q_heads, G)) return S3R_ERR_CUDA;
    a.test_stall = g_test_stall.exchange(0);
    return to_status(launch_verify_tc(kmap, vmap, qmap, a, sms, static_cast<cudaStream_t>(stream)));
  }
  return to_status(launch_attention(kmap, vmap, a, sms, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

const char* s3r_version(void) { return "s3r-b300 0.1.0 (sm_103a)"; }

void s3r_test_stall_next_verify(void) { g_test_stall.store(1); }

const char* s3r_status_string(s3r_status status) {
  switch (status) {
    case S3R_OK: return "S3R_OK";
    case S3R_ERR_INVALID_ARG: return "S3R_ERR_INVALID_ARG";
    case S3R_ERR_UNSUPPORTED: return "S3R_ERR_UNSUPPORTED";
    case S3R_ERR_CUDA: return "S3R_ERR_CUDA";
    case S3R_ERR_WORKSPACE: return "S3R_ERR_WORKSPACE";
  }
  return "S3R_UNKNOWN_STATUS";
}

s3r_status s3r_attn_workspace_size(const s3r_paged_kv* kv, int32_t max_block_rows, size_t* bytes) {
  if (bytes == nullptr) return S3R_ERR_INVALID_ARG;
  s3r_status st = validate_kv(kv);
  if (st != S3R_OK) return st;
  if (max_block_rows <= 0) return S3R_ERR_INVALID_ARG;
  const int G = kv->num_q_heads / kv->num_kv_heads;
  const int64_t R = static_cast<int64_t>(max_block_rows) * G;
  if (R > S3R_MAX_ROWS_PER_KV_HEAD) return S3R_ERR_UNSUPPORTED;
  const int sms = current_sm_count();
  if (sms <= 0) return S3R_ERR_CUDA;
  *bytes = attn_workspace_layout(kv->num_seqs * kv->num_kv_heads, static_cast<int>(R),
                                 kv->max_pages_per_seq, sms * kAttnWarps, true)
               .total;
  return S3R_OK;
}

s3r_status s3r_spec_sample_workspace_size(int32_t n, int32_t k, size_t* bytes) {
  if (bytes == nullptr || n < 0 || k < 0) return S3R_ERR_INVALID_ARG;
  if (k > kMaxSpecK) return S3R_ERR_UNSUPPORTED;
  *bytes = spec_workspace_layout(n, k).total;
  return S3R_OK;
}

s3r_status s3r_select_workspace_size(size_t* bytes) {
  if (bytes == nullptr) return S3R_ERR_INVALID_ARG;
  *bytes = 256;
  return S3R_OK;
}

s3r_status s3r_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || !aligned256(ws) || ws_bytes < 256) return S3R_ERR_WORKSPACE;
  return to_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

s3r_status s3r_read_device_error(const void* ws, void* stream, int32_t* code, int32_t clear) {
  if (ws == nullptr || code == nullptr) return S3R_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return S3R_ERR_CUDA;
  *code = v;
  if (clear) {
    e = cudaMemsetAsync(const_cast<void*>(ws), 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return S3R_ERR_CUDA;
  }
  return S3R_OK;
}

s3r_status s3r_dense_decode_attn(const s3r_paged_kv* kv, const int32_t* ctx_lens, const void* q,
                                 void* out, float sm_scale, void* ws, size_t ws_bytes,
                                 void* stream) {
  return run_attention(kv, kModeDense, ctx_lens, 1, 0, nullptr, nullptr, 0, q, out, nullptr, 0,
                       sm_scale, ws, ws_bytes, stream);
}

s3r_status s3r_sparse_draft_attn(const s3r_paged_kv* kv, const int32_t* hist_lens,
                                 int32_t draft_pos, const int32_t* sel_pages,
                                 const int32_t* sel_count, int32_t b_max, const void* q, void* out,
                                 float sm_scale, void* ws, size_t ws_bytes, void* stream) {
  return run_attention(kv, kModeSparse, hist_lens, 1, draft_pos, sel_pages, sel_count, b_max, q,
                       out, nullptr, 0, sm_scale, ws, ws_bytes, stream);
}

s3r_status s3r_verify_attn(const s3r_paged_kv* kv, const int32_t* hist_lens, int32_t n_rows,
                           const void* q, void* out, float* page_mass, int32_t mass_stride,
                           float sm_scale, void* ws, size_t ws_bytes, void* stream) {
  return run_attention(kv, kModeVerify, hist_lens, n_rows, 0, nullptr, nullptr, 0, q, out,
                       page_mass, mass_stride, sm_scale, ws, ws_bytes, stream);
}

s3r_status s3r_dense_decode_attn_append(const s3r_paged_kv* kv, const int32_t* ctx_lens, const s3r_kv_rows* rows,
                                        const void* q, void* out, float sm_scale, void* ws, size_t ws_bytes,
                                        void* stream) {
  if (rows == nullptr) return S3R_ERR_INVALID_ARG;
  return run_attention(kv, kModeDense, ctx_lens, 1, 0, nullptr, nullptr, 0, q, out, nullptr, 0, sm_scale, ws,
                       ws_bytes, stream, rows);
}

s3r_status s3r_sparse_draft_attn_append(const s3r_paged_kv* kv, const int32_t* hist_lens, int32_t draft_pos,
                                        const int32_t* sel_pages, const int32_t* sel_count, int32_t b_max,
                                        const s3r_kv_rows* rows, const void* q, void* out, float sm_scale,
                                        void* ws, size_t ws_bytes, void* stream) {
  if (rows == nullptr) return S3R_ERR_INVALID_ARG;
  return run_attention(kv, kModeSparse, hist_lens, 1, draft_pos, sel_pages, sel_count, b_max, q, out, nullptr, 0,
                       sm_scale, ws, ws_bytes, stream, rows);
}

s3r_status s3r_verify_attn_append(const s3r_paged_kv* kv, const int32_t* hist_lens, int32_t n_rows,
                                  const s3r_kv_rows* rows, const void* q, void* out, float* page_mass,
                                  int32_t mass_stride, float sm_scale, void* ws, size_t ws_bytes, void* stream) {
  if (rows == nullptr) return S3R_ERR_INVALID_ARG;
  return run_attention(kv, kModeVerify, hist_lens, n_rows, 0, nullptr, nullptr, 0, q, out, page_mass, mass_stride,
                       sm_scale, ws, ws_bytes, stream, rows);
}

s3r_status s3r_select_draft_pages(const float* page_mass, const int32_t* sel_lens, int32_t num_seqs,
                                  int32_t num_kv_heads, int32_t mass_stride, double budget,
                                  int32_t n_sink, int32_t n_recent, int32_t* sel_pages,
                                  int32_t* sel_count, int32_t b_max, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (num_seqs < 0 || num_kv_heads <= 0 || mass_stride <= 0 || n_sink < 0 || n_recent < 0 ||
      b_max < 0)
    return S3R_ERR_INVALID_ARG;
  if (!(budget >= 0.0 && budget <= 1.0)) return S3R_ERR_INVALID_ARG;
  if (mass_stride > kMaxSelectPages) return S3R_ERR_UNSUPPORTED;
  if (ws == nullptr || !aligned256(ws) || ws_bytes < 256) return S3R_ERR_WORKSPACE;
  if (static_cast<int64_t>(num_seqs) * num_kv_heads > 0x7fffffff) return S3R_ERR_UNSUPPORTED;
  if (num_seqs == 0) return S3R_OK;
  if (page_mass == nullptr || sel_lens == nullptr || sel_pages == nullptr || sel_count == nullptr)
    return S3R_ERR_INVALID_ARG;
  // The page budget grows with the history; the longest history the mass
  // rows can describe is mass_stride pages.
  const int P = mass_stride;
  const int n_mand = std::min(n_sink, P) + (P - std::max(std::max(P - n_recent, 0), std::min(n_sink, P)));
  const double want = std::ceil(budget * static_cast<double>(P) - 1e-9);
  const int B = static_cast<int>(std::min(static_cast<double>(P), std::max(want, static_cast<double>(n_mand))));
  if (b_max < B) return S3R_ERR_INVALID_ARG;
  return to_status(launch_select_pages(page_mass, sel_lens, num_seqs, num_kv_heads, mass_stride,
                                       budget, n_sink, n_recent, sel_pages, sel_count, b_max,
                                       static_cast<int*>(ws), static_cast<cudaStream_t>(stream)));
}

static s3r_status check_spec_sample(const float* p_logits, const float* q_logits, const int32_t* draft_tokens,
                                     int32_t n, int32_t k, int32_t vocab, uint64_t offset, int32_t* out_tokens,
                                     int32_t* n_accepted, void* ws, size_t ws_bytes) {
  const s3r_status st =
      s3r::check_spec_sample_args(p_logits, q_logits, draft_tokens, n, k, vocab, offset, out_tokens, n_accepted);
  if (st != S3R_OK) return st;
  size_t need = 0;
  s3r_spec_sample_workspace_size(n, k, &need);
  if (ws == nullptr || !aligned256(ws) || ws_bytes < need) return S3R_ERR_WORKSPACE;
  return S3R_OK;
}

// Zero the optional tie counters before the sampler kernels add to them.
static s3r_status zero_ties(uint32_t* tie_count, cudaStream_t stream) {
  if (tie_count == nullptr) return S3R_OK;
  return to_status(cudaMemsetAsync(tie_count, 0, 2 * sizeof(uint32_t), stream));
}

s3r_status s3r_spec_sample(const float* p_logits, const float* q_logits,
                           const int32_t* draft_tokens, int32_t n, int32_t k, int32_t vocab,
                           uint64_t seed, uint64_t offset, int32_t* out_tokens,
                           int32_t* n_accepted, uint32_t* tie_count, void* ws, size_t ws_bytes, void* stream) {
  s3r_status st = check_spec_sample(p_logits, q_logits, draft_tokens, n, k, vocab, offset, out_tokens,
                                    n_accepted, ws, ws_bytes);
  if (st != S3R_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = zero_ties(tie_count, s);
  if (st != S3R_OK || n == 0) return st;
  return to_status(launch_spec_sample(p_logits, q_logits, draft_tokens, n, k, vocab, seed,
                                      static_cast<uint32_t>(offset), ws, out_tokens, n_accepted, s, 1, -1, 0, 1,
                                      tie_count));
}

s3r_status s3r_spec_sample_sequential(const float* p_logits, const float* q_logits,
                                      const int32_t* draft_tokens, int32_t n, int32_t k, int32_t vocab,
                                      uint64_t seed, uint64_t offset, int32_t* out_tokens,
                                      int32_t* n_accepted, uint32_t* tie_count, void* ws, size_t ws_bytes,
                                      void* stream) {
  s3r_status st = check_spec_sample(p_logits, q_logits, draft_tokens, n, k, vocab, offset, out_tokens,
                                    n_accepted, ws, ws_bytes);
  if (st != S3R_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = zero_ties(tie_count, s);
  if (st != S3R_OK || n == 0) return st;
  return to_status(launch_spec_sample_sequential(p_logits, q_logits, draft_tokens, n, k, vocab, seed,
                                                 static_cast<uint32_t>(offset), ws, out_tokens, n_accepted, s,
                                                 tie_count));
}

s3r_status s3r_sample_draft_tokens(const float* logits, int32_t n, int32_t vocab, int64_t row_stride,
                                   uint64_t seed, uint64_t offset, int32_t draft_pos, int32_t* tokens,
                                   int64_t token_stride, void* ws, size_t ws_bytes, void* stream) {
  if (n < 0 || vocab <= 0 || draft_pos < 0 || row_stride < vocab || token_stride < 1) return S3R_ERR_INVALID_ARG;
  if (offset > 0xffffffffULL) return S3R_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n) * row_stride > (int64_t{1} << 40)) return S3R_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(n) * kSampleChunks > 0x7fffffffLL) return S3R_ERR_UNSUPPORTED;
  size_t need = 0;
  s3r_sample_draft_workspace_size(n, &need);
  if (ws == nullptr || !aligned256(ws) || ws_bytes < need) return S3R_ERR_WORKSPACE;
  if (n == 0) return S3R_OK;
  if (logits == nullptr || tokens == nullptr) return S3R_ERR_INVALID_ARG;
  const SpecWorkspaceLayout L = spec_workspace_layout(n, 0);
  int32_t* count = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + L.accept_off);
  return to_status(launch_spec_sample(logits, nullptr, nullptr, n, 0, vocab, seed, static_cast<uint32_t>(offset),
                                      ws, tokens, count, static_cast<cudaStream_t>(stream), kStreamDraftU,
                                      draft_pos, row_stride, token_stride));
}

s3r_status s3r_sample_draft_workspace_size(int32_t n, size_t* bytes) {
  if (bytes == nullptr || n < 0) return S3R_ERR_INVALID_ARG;
  *bytes = spec_workspace_layout(n, 0).total;
  return S3R_OK;
}

s3r_status s3r_kv_append(const s3r_paged_kv* kv, const int32_t* start_lens, const int32_t* n_rows,
                         int32_t max_rows, const void* k_rows, const void* v_rows, void* ws, size_t ws_bytes,
                         void* stream) {
  const s3r_status st = validate_kv(kv);
  if (st != S3R_OK) return st;
  if (max_rows < 0) return S3R_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned256(ws) || ws_bytes < 256) return S3R_ERR_WORKSPACE;
  if (static_cast<int64_t>(kv->num_seqs) * max_rows > 0x7fffffffLL) return S3R_ERR_UNSUPPORTED;
  if (kv->num_seqs == 0 || max_rows == 0) return S3R_OK;
  if (start_lens == nullptr || k_rows == nullptr || v_rows == nullptr) return S3R_ERR_INVALID_ARG;
  if (!aligned16(k_rows) || !aligned16(v_rows)) return S3R_ERR_INVALID_ARG;
  KvAppendArgs a{};
  // the pools are declared const in s3r_paged_kv because attention only reads them
  a.k_pool = const_cast<void*>(kv->k_pool);
  a.v_pool = const_cast<void*>(kv->v_pool);
  a.block_table = kv->block_table;
  a.num_phys_pages = kv->num_phys_pages;
  a.max_pages = kv->max_pages_per_seq;
  a.S = kv->num_seqs;
  a.Hkv = kv->num_kv_heads;
  a.start_lens = start_lens;
  a.n_rows = n_rows;
  a.max_rows = max_rows;
  a.k_rows = k_rows;
  a.v_rows = v_rows;
  a.err = static_cast<int*>(ws);
  return to_status(launch_kv_append(a, static_cast<cudaStream_t>(stream)));
}

s3r_status s3r_commit_lengths(const int32_t* hist_lens, const int32_t* n_accepted, int32_t n, int32_t max_accept,
                              int32_t max_len, int32_t* new_lens, void* ws, size_t ws_bytes, void* stream) {
  if (n < 0 || max_accept < 0 || max_len < 0) return S3R_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned256(ws) || ws_bytes < 256) return S3R_ERR_WORKSPACE;
  if (n == 0) return S3R_OK;
  if (hist_lens == nullptr || n_accepted == nullptr || new_lens == nullptr) return S3R_ERR_INVALID_ARG;
  return to_status(launch_commit_lengths(hist_lens, n_accepted, n, max_accept, max_len, new_lens,
                                         static_cast<int*>(ws), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

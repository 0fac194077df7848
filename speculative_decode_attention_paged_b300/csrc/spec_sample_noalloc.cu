// s3r_spec_sample_noalloc: exact speculative sampling for callers that cannot
// allocate device memory.
//
// Some callers have no way to allocate a workspace: code running inside a
// memory pool that is fully reserved up front, plugins handed only their
// input and output buffers, or drivers that forbid cudaMalloc after start-up.
// This entry point runs the same sampler as s3r_spec_sample (row statistics,
// ratio tests, residual chunk sums and the inverse-CDF pick in one launch; for
// k = 0 the one-pass bonus sampler), with its scratch (the error word, the
// per-row statistics, the per-sequence counters and the task ticket) in a
// fixed-size array that lives in the library's own device image.  The array exists once
// per GPU that loads the library and stays allocated until the process exits.
//
// The array is a __device__ symbol: in host code its name is only a host-side
// stand-in, so the device address is looked up once per device with
// cudaGetSymbolAddress and cached.  Nothing here calls cudaMalloc, cudaFree or
// an allocating library routine.

#include <mutex>

#include "../../include/s3r.h"
#include "spec_sample.cuh"

#include <cuda_runtime.h>

namespace {

constexpr int kMaxDevices = 64;

// Scratch of every s3r_spec_sample_noalloc call on this device: the first 256
// bytes are the device error word, the rest holds the row statistics.
static __device__ __align__(256) unsigned char g_noalloc_scratch[S3R_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call per device), or null on failure.
void* scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

// Forget the cached address after a CUDA failure, so that the next call looks
// it up again instead of reusing an address a reset may have invalidated.
s3r_status forget_on_failure(int dev, s3r_status st) {
  if (st == S3R_ERR_CUDA) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    g_scratch_ptr[dev] = nullptr;
  }
  return st;
}

}  // namespace

extern "C" s3r_status s3r_spec_sample_noalloc(const float* p_logits, const float* q_logits,
                                              const int32_t* draft_tokens, int32_t n, int32_t k,
                                              int32_t vocab, uint64_t seed, uint64_t offset,
                                              int32_t* out_tokens, int32_t* n_accepted,
                                              int32_t* device_error, void* stream) {
  // The size limit and every argument check run before the shared scratch is
  // touched, so a rejected call enqueues nothing (not even the clears below).
  size_t need = 0;
  s3r_status st = s3r_spec_sample_workspace_size(n, k, &need);
  if (st != S3R_OK) return st;
  if (need > S3R_NOALLOC_SCRATCH_BYTES) return S3R_ERR_UNSUPPORTED;
  st = s3r::check_spec_sample_args(p_logits, q_logits, draft_tokens, n, k, vocab, offset, out_tokens, n_accepted);
  if (st != S3R_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return S3R_ERR_CUDA;
  void* ws = scratch_address(dev);
  if (ws == nullptr) return S3R_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: clear the error word and
  // the counters the sampler's kernels count on (per-sequence arrivals and
  // flags, the task ticket), which a call that stopped on a device error may
  // have left set.
  if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return forget_on_failure(dev, S3R_ERR_CUDA);
  if (n > 0) {
    const s3r::SpecWorkspaceLayout L = s3r::spec_workspace_layout(n, k);
    if (cudaMemsetAsync(static_cast<unsigned char*>(ws) + L.arrive_off, 0, L.total - L.arrive_off, s) != cudaSuccess)
      return forget_on_failure(dev, S3R_ERR_CUDA);
  }
  st = s3r_spec_sample(p_logits, q_logits, draft_tokens, n, k, vocab, seed, offset, out_tokens, n_accepted,
                       nullptr, ws, S3R_NOALLOC_SCRATCH_BYTES, stream);
  if (st != S3R_OK) return forget_on_failure(dev, st);
  if (device_error != nullptr &&
      cudaMemcpyAsync(device_error, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return forget_on_failure(dev, S3R_ERR_CUDA);
  return S3R_OK;
}

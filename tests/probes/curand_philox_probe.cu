// Test helper: evaluates CUDA's curand Philox4x32-10 device routine on given
// (counter, key) pairs, so the oracle's Philox can be pinned against a library
// implementation of the same published generator.  Not part of the library.
#include <cstdint>
#include <cuda_runtime.h>
#include <curand_kernel.h>

namespace {
__global__ void philox_probe_kernel(const uint4* ctr, const uint2* key, uint4* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = curand_Philox4x32_10(ctr[i], key[i]);
}
}  // namespace

extern "C" __attribute__((visibility("default"))) int philox_probe_run(const void* ctr, const void* key,
                                                                       void* out, int n, void* stream) {
  if (n <= 0) return 0;
  philox_probe_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(ctr), static_cast<const uint2*>(key), static_cast<uint4*>(out), n);
  return static_cast<int>(cudaGetLastError());
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11, section 3.2): ten rounds of the 4x32 Philox bijection,
// each round two 32x32->64 multiplies (multipliers 0xD2511F53, 0xCD9E8D57)
// whose halves are xored with the other words and the round key, the key
// bumped between rounds by the Weyl increments 0x9E3779B9 and 0xBB67AE85.
#pragma once

#include <cstdint>

namespace s3r {

enum PhiloxStream : uint32_t { kStreamAccept = 0, kStreamResample = 1, kStreamDraft = 2 };

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// Uniform in [0, 1) on the 2^-24 grid for counter (n, pos, stream, offset),
// key = (seed low word, seed high word).
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t offset, uint32_t n,
                                                uint32_t pos, uint32_t stream) {
  const uint4 r = philox4x32_10(make_uint4(n, pos, stream, offset),
                                make_uint2(static_cast<uint32_t>(seed),
                                           static_cast<uint32_t>(seed >> 32)));
  return static_cast<float>(r.x >> 8) * 5.9604644775390625e-08f;   // 2^-24
}

}  // namespace s3r

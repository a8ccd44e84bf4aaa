// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC'11, section 4.2): ten rounds of the Philox-4x32 S-box with the
// multipliers 0xD2511F53 / 0xCD9E8D57 and the Weyl key increments 0x9E3779B9 /
// 0xBB67AE85.  Device implementation for the selector walk and the verify draws.
//
// Stream layout of the step: key = (seed lo32, seed hi32), counter = (offset lo32,
// offset hi32, slot, purpose); u = (x0 >> 8) * 2^-24.
#pragma once
#include <stdint.h>

namespace df2 {

enum : uint32_t { kPurposeWalk = 0, kPurposeAccept = 1, kPurposeResample = 2 };

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ float philox_uniform(uint64_t seed, uint64_t offset, uint32_t slot, uint32_t purpose) {
  const uint4 c = make_uint4(static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32), slot, purpose);
  const uint2 k = make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const uint4 o = philox4x32_10(c, k);
  return static_cast<float>(o.x >> 8) * (1.0f / 16777216.0f);
}

}  // namespace df2

// Philox4x32-10 counter-based generator, device side.
//
// J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random numbers:
// as easy as 1, 2, 3", SC'11: each of the 10 rounds multiplies counter words 0
// and 2 by the two round multipliers, XORs the high product halves with words
// 1 and 3 and the round key, and the key advances by the two Weyl increments.
// Only word 0 of the output is used here.
#pragma once
#include <cstdint>

namespace sv {

__device__ __forceinline__ uint32_t philox4x32_10_word0(uint32_t c0, uint32_t c1, uint32_t c2,
                                                        uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c0;
}

// U(seed, s, pos, draw) in [0, 1): key = (seed lo, seed hi), counter =
// (s lo, pos, draw, s hi), the top 24 bits of output word 0 times 2^-24
// (exact in float).
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint64_t s, uint32_t pos,
                                                uint32_t draw) {
  const uint32_t x = philox4x32_10_word0(static_cast<uint32_t>(s), pos, draw,
                                         static_cast<uint32_t>(s >> 32),
                                         static_cast<uint32_t>(seed),
                                         static_cast<uint32_t>(seed >> 32));
  return static_cast<float>(x >> 8) * 0x1p-24f;
}

}  // namespace sv

// rng.cuh -- the random numbers of sampling mode: Philox4x32-10 (Salmon,
// Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11),
// key (seed low, seed high), counter (entry, position, sequence << 8 |
// purpose, cycle); u = ((x0 >> 8) + 1/2) 2^-24 in (0, 1); g = -log(-log u)
// a Gumbel(0, 1) variate.  The purposes keep the draws of the different
// decisions apart.
#pragma once
#include <stdint.h>

namespace dfl {

enum : uint32_t { RNG_DRAFT = 1, RNG_ACCEPT = 2, RNG_RESID = 3, RNG_BONUS = 4, RNG_PATH = 5 };

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

__device__ __forceinline__ float rng_uniform(uint64_t seed, uint32_t v, uint32_t pos, uint32_t seq, uint32_t purpose,
                                             uint32_t cycle) {
  const uint4 x = philox4x32_10(make_uint4(v, pos, (seq << 8) | (purpose & 0xFFu), cycle), (uint32_t)seed,
                                (uint32_t)(seed >> 32));
  return ((float)(x.x >> 8) + 0.5f) * (1.0f / 16777216.0f);
}

__device__ __forceinline__ float rng_gumbel(uint64_t seed, uint32_t v, uint32_t pos, uint32_t seq, uint32_t purpose,
                                            uint32_t cycle) {
  return -logf(-logf(rng_uniform(seed, v, pos, seq, purpose, cycle)));
}

}  // namespace dfl

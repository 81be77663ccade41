// Philox4x32-10 counter-based generator, device side.
//
// From the definition in Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3" (SC'11): four 32-bit counter words, two key
// words; each round multiplies words 0 and 2 by fixed odd constants, takes
// the 64-bit products apart into high and low halves, mixes the high halves
// with the other two words and the key, and the key advances by the Weyl
// increments between rounds.  Ten rounds.
#pragma once
#include <cstdint>

namespace attn {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// The key of each of the ten rounds: (seed_lo + r W0, seed_hi + r W1) mod 2^32.
// The host fills it once per call, so the rounds read their keys from kernel
// parameters instead of re-deriving them in every call.
struct PhiloxRoundKeys {
  uint32_t k0[10], k1[10];
};

__host__ __device__ inline PhiloxRoundKeys philox_round_keys(uint32_t seed_lo, uint32_t seed_hi) {
  PhiloxRoundKeys rk{};
  for (uint32_t r = 0; r < 10; ++r) {
    rk.k0[r] = seed_lo + r * kPhiloxW0;
    rk.k1[r] = seed_hi + r * kPhiloxW1;
  }
  return rk;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxRoundKeys& rk) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(kPhiloxM0) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(kPhiloxM1) * c.z;
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
    c = make_uint4(hi1 ^ c.y ^ rk.k0[r], lo1, hi0 ^ c.w ^ rk.k1[r], lo0);
  }
  return c;
}

// Keep bits of four consecutive keys j = 4g .. 4g+3 of query row i:
// bit t of the result is 1 iff key 4g+t is kept (word t >= threshold).
__device__ __forceinline__ uint32_t dropout_keep4(uint32_t g, uint32_t i, uint32_t bh,
                                                  uint32_t offset, const PhiloxRoundKeys& rk,
                                                  uint32_t threshold) {
  const uint4 u = philox4x32_10(make_uint4(g, i, bh, offset), rk);
  return (u.x >= threshold ? 1u : 0u) | (u.y >= threshold ? 2u : 0u) |
         (u.z >= threshold ? 4u : 0u) | (u.w >= threshold ? 8u : 0u);
}

// Keep bits of the 32 query rows q0 .. q0+31 for key kj, where the four
// lanes of an aligned lane quad hold the four keys 4g .. 4g+3 (kj mod 4 ==
// lane mod 4).  One Philox call at query q yields the words of all four
// keys, so each lane evaluates the 8 queries q0 + 4s + (lane mod 4) and the
// quad exchanges the results: 8 calls per lane instead of 32.  Bit t of the
// result is 1 iff (q0 + t, kj) is kept.  All 32 lanes must call it.
__device__ __forceinline__ uint32_t dropout_keep32_by_key(uint32_t kj, uint32_t q0, uint32_t bh,
                                                          uint32_t offset,
                                                          const PhiloxRoundKeys& rk,
                                                          uint32_t threshold, uint32_t lane) {
  const uint32_t u = lane & 3u;
  uint32_t mine = 0;   // bit 4s + x: key 4g+x kept at query q0 + 4s + u
#pragma unroll
  for (uint32_t s = 0; s < 8; ++s)
    mine |= dropout_keep4(kj >> 2, q0 + 4 * s + u, bh, offset, rk, threshold) << (4 * s);
  uint32_t keep = 0;
#pragma unroll
  for (uint32_t src = 0; src < 4; ++src) {
    const uint32_t m = __shfl_sync(0xffffffffu, mine, (lane & ~3u) | src);
#pragma unroll
    for (uint32_t s = 0; s < 8; ++s) keep |= ((m >> (4 * s + u)) & 1u) << (4 * s + src);
  }
  return keep;
}

}  // namespace attn

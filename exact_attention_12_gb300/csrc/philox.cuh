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

// Shifts the keep bits of one Philox output into `acc`, most significant key
// first: word w holds the 16-bit uniforms of keys 2w (low half) and 2w+1
// (high half) of its group of eight, and a key is kept iff its uniform is at
// least the threshold T (1 <= T <= 65535).  With k16 = (2^16 - T) << 16, a
// half h is >= T exactly when (h << 16) + k16 carries out of 32 bits, and
// the carry is shifted in by acc + acc + carry.  Afterwards the low eight
// bits of acc hold keys 0..7 of the group (bit t = key t).
__device__ __forceinline__ uint32_t push_keep8(uint32_t acc, uint4 u, uint32_t k16) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 3; k >= 0; --k)
    asm("{\n\t.reg .u32 t;\n\t"
        "add.cc.u32 t, %1, %2;\n\t"     // high half (key 2k+1)
        "addc.u32 %0, %0, %0;\n\t"
        "shl.b32 t, %1, 16;\n\t"
        "add.cc.u32 t, t, %2;\n\t"      // low half (key 2k)
        "addc.u32 %0, %0, %0;\n\t}"
        : "+r"(acc)
        : "r"(w[k]), "r"(k16));
  return acc;
}

__device__ __forceinline__ uint32_t keep_k16(uint32_t threshold) {
  return (0x10000u - threshold) << 16;
}

// Keep bits of eight consecutive keys j = 8g .. 8g+7 of query row i: bit t
// of the result is 1 iff key 8g+t is kept.
__device__ __forceinline__ uint32_t dropout_keep8(uint32_t g, uint32_t i, uint32_t bh,
                                                  uint32_t offset, const PhiloxRoundKeys& rk,
                                                  uint32_t threshold) {
  return push_keep8(0u, philox4x32_10(make_uint4(g, i, bh, offset), rk), keep_k16(threshold));
}

// Keep bits of the 32 keys j = 8g .. 8g+31 of query row i (four Philox
// calls): bit t of the result is 1 iff key 8g+t is kept.
__device__ __forceinline__ uint32_t dropout_keep32(uint32_t g, uint32_t i, uint32_t bh,
                                                   uint32_t offset, const PhiloxRoundKeys& rk,
                                                   uint32_t threshold) {
  uint4 u[4];
#pragma unroll
  for (uint32_t s = 0; s < 4; ++s) u[s] = philox4x32_10(make_uint4(g + s, i, bh, offset), rk);
  const uint32_t k16 = keep_k16(threshold);
  uint32_t acc = 0;
#pragma unroll
  for (int s = 3; s >= 0; --s) acc = push_keep8(acc, u[s], k16);
  return acc;
}

// Keep bits of the 32 query rows q0 .. q0+31 for key kj, where the eight
// lanes of an aligned lane octet hold the keys 8g .. 8g+7 (kj mod 8 ==
// lane mod 8).  One Philox call at query q yields the uniforms of all eight
// keys, so each lane evaluates the 4 queries q0 + 8s + (lane mod 8): byte s
// of its word holds the keep bits of keys 8g .. 8g+7 at that query.  Per
// byte, the octet then holds an 8 x 8 bit matrix (row = lane, column = key)
// and each lane needs one column: three butterfly stages transpose it, each
// exchanging words with lane ^ k (k = 4, 2, 1) and swapping the off-diagonal
// k x k bit blocks (the recursive block transpose; all four bytes at once).
// Bit t of the result is 1 iff (q0 + t, kj) is kept.  All 32 lanes must call it.
__device__ __forceinline__ uint32_t dropout_keep32_by_key(uint32_t kj, uint32_t q0, uint32_t bh,
                                                          uint32_t offset,
                                                          const PhiloxRoundKeys& rk,
                                                          uint32_t threshold, uint32_t lane) {
  const uint32_t u = lane & 7u;
  uint32_t x = 0;
#pragma unroll
  for (uint32_t s = 0; s < 4; ++s)
    x |= dropout_keep8(kj >> 3, q0 + 8 * s + u, bh, offset, rk, threshold) << (8 * s);
  constexpr uint32_t kHigh[3] = {0xF0F0F0F0u, 0xCCCCCCCCu, 0xAAAAAAAAu};
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const uint32_t k = 4u >> i;
    const uint32_t p = __shfl_xor_sync(0xffffffffu, x, static_cast<int>(k));
    x = (u & k) ? ((x & kHigh[i]) | ((p >> k) & ~kHigh[i]))
                : ((x & ~kHigh[i]) | ((p << k) & kHigh[i]));
  }
  return x;
}

}  // namespace attn

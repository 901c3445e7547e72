// Philox4x64-10 counter-based generator (Salmon, Moraes, Dror, Shaw 2011,
// "Parallel random numbers: as easy as 1, 2, 3", §4) and the LoRA dropout
// mask drawn from it.
#pragma once

#include <cstdint>

namespace lora {

// Four 64-bit counter words and two key words in, four words out: each of
// the 10 rounds multiplies words 0 and 2 by the round multipliers and mixes
// the halves of the products with words 1 and 3 and the key; the key
// advances by the two Weyl increments between rounds.
struct Philox4x64 {
  uint64_t v[4];
  __device__ __forceinline__ Philox4x64(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3,
                                        uint64_t k0, uint64_t k1) {
    constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
    constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
      if (r > 0) {
        k0 += kW0;
        k1 += kW1;
      }
      const uint64_t hi0 = __umul64hi(kM0, c0), lo0 = kM0 * c0;
      const uint64_t hi1 = __umul64hi(kM1, c2), lo1 = kM1 * c2;
      const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
      c0 = n0;
      c1 = lo1;
      c2 = n2;
      c3 = lo0;
    }
    v[0] = c0;
    v[1] = c1;
    v[2] = c2;
    v[3] = c3;
  }
};

// LoRA dropout mask of x [M, k] (row-major element e = i·k + j): element e
// takes 16-bit number e mod 16 of the block with counter (e / 16, offset, 0,
// 0) and key (seed, 0), the four output words read as sixteen 16-bit numbers
// low half first, and is kept iff that number is at least `thresh`
// (round(p·65536)).  Returns the 16 keep bits of block b (bit i: element
// 16·b + i).
__device__ __forceinline__ uint32_t dropout_keep16(uint64_t b, uint64_t seed, uint64_t offset,
                                                   uint32_t thresh) {
  const Philox4x64 ph(b, offset, 0ull, 0ull, seed, 0ull);
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t u = (uint32_t)(ph.v[i >> 2] >> (16 * (i & 3))) & 0xFFFFu;
    bits |= (u >= thresh ? 1u : 0u) << i;
  }
  return bits;
}

}  // namespace lora

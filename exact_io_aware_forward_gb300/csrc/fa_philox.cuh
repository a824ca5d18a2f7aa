// Philox4x32-10 counter-based generator for attention dropout, written from
// its published definition (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC 2011).  The dropout passage of
// "FlashAttention 为什么不需要存下注意力矩阵" (jefxiong.cn), section 05, keeps
// only the generator's seed and offset: the backward pass draws the same
// keep mask again instead of reading a stored one.
//
// Counter mapping (one call per 8 consecutive keys of one query row):
// entry (head bh, query i, key j) uses counter (j / 8, i, bh, offset) under
// key (seed low word, seed high word); output word (j / 2) % 4 holds the
// 16-bit draw of key j in its low half (j even) or high half (j odd); the
// entry is kept iff draw >= t, with t = round(p * 65536).
#pragma once

#include <stdint.h>

namespace fa {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;  // golden ratio, 32-bit fixed point
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;  // sqrt(3) - 1, 32-bit fixed point

// Ten rounds: multiply words 0 and 2, mix the high halves into words 1 and 3
// with the round key, permute; the key advances by the Weyl constants.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)kPhiloxM0 * c.x;
    const uint64_t p1 = (uint64_t)kPhiloxM1 * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0);
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return c;
}

// 0xffff in each 16-bit half of w whose draw is kept (>= t), 0 elsewhere: a
// mask that zeroes the dropped element of a packed 16-bit pair.
__device__ __forceinline__ uint32_t keep_halves(uint32_t w, uint32_t t) {
  const uint32_t lo = (w & 0xffffu) >= t ? 0x0000ffffu : 0u;
  const uint32_t hi = (w >> 16) >= t ? 0xffff0000u : 0u;
  return lo | hi;
}

// Keep bits of the 8 keys of one generator call: bit k <-> key 8 * (j / 8) + k.
__device__ __forceinline__ uint32_t keep_byte(uint4 w, uint32_t t) {
  uint32_t b = 0;
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    b |= ((ws[r] & 0xffffu) >= t ? 1u : 0u) << (2 * r);
    b |= ((ws[r] >> 16) >= t ? 1u : 0u) << (2 * r + 1);
  }
  return b;
}

}  // namespace fa

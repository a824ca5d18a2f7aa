// Philox4x32-10 counter-based generator for attention dropout, written from
// its published definition (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC 2011).  The dropout passage of
// "FlashAttention 为什么不需要存下注意力矩阵" (jefxiong.cn), section 05, keeps
// only the generator's seed and offset: the backward pass draws the same
// keep mask again instead of reading a stored one.
//
// Counter mapping (one call per 16 consecutive keys of one query row):
// entry (head bh, query i, key j) uses counter (j / 16, i, bh, offset) under
// key (seed low word, seed high word); output word (j / 4) % 4 holds the
// 8-bit draw of key j in its byte j % 4 (least significant first); the entry
// is kept iff draw >= t, with t = round(p * 256).
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

// Keep bits of the 16 keys of one generator call: bit k <-> key 16 * (j / 16) + k.
// `tt` is t in each of the four bytes; __vsetgeu4 gives 1 in bit 0 of each
// byte whose draw is >= t, and the shifts gather those four bits.
__device__ __forceinline__ uint32_t keep_bits16(uint4 w, uint32_t tt) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t b = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t v = __vsetgeu4(ws[r], tt);
    b |= ((v | (v >> 7) | (v >> 14) | (v >> 21)) & 0xFu) << (4 * r);
  }
  return b;
}

// Keep bits of the 32 * NW keys [kbase, kbase + 32 NW) of query `row`, one
// word per 32 keys: in word cc, bit i is the even key kbase + 32cc + 2i of
// pair i and bit 16 + i the odd key kbase + 32cc + 2i + 1 (2 NW generator
// calls; kbase a multiple of 32).
template <int NW>
__device__ __forceinline__ void tile_keep_bits(uint32_t (&eo)[NW], int kbase, int row, int bh, uint32_t offset,
                                               uint32_t k0, uint32_t k1, uint32_t t) {
  const uint32_t tt = t * 0x01010101u;
#pragma unroll
  for (int cc = 0; cc < NW; ++cc) {
    uint32_t e = 0;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const uint4 w = philox4x32_10(
          make_uint4(((uint32_t)(kbase + 32 * cc) >> 4) + g, (uint32_t)row, (uint32_t)bh, offset), k0, k1);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        // Word r holds keys 16g + 4r + {0, 1, 2, 3}: the even and odd keys of
        // pairs 8g + 2r and 8g + 2r + 1.  With v's bits at 0, 8, 16, 24, u has
        // key +0 at bit 0, key +2 at bit 1, key +1 at bit 8, key +3 at bit 9.
        const uint32_t v = __vsetgeu4(ws[r], tt);
        const uint32_t u = v | (v >> 15);
        e |= ((u & 0x3u) | ((u & 0x300u) << 8)) << (8 * g + 2 * r);
      }
    }
    eo[cc] = e;
  }
}

// 0xffff over each kept half of packed pair i from a keep word of
// tile_keep_bits: bits i and 16 + i are moved to bits 7 and 23, and prmt
// replicates the top bit of bytes 0 and 2 over the low and high halves.
__device__ __forceinline__ uint32_t pair_keep_mask(uint32_t eo, int i) {
  const uint32_t x = i <= 7 ? eo << (7 - i) : eo >> (i - 7);
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, 0xAA88;" : "=r"(m) : "r"(x));
  return m;
}

// One step of a bit-matrix transpose across lanes: rows are lanes, columns
// are bits; partners lane ^ m swap the off-diagonal m x m blocks (lo_mask
// selects the low block of every 2m-bit group).
__device__ __forceinline__ uint32_t transpose_step(uint32_t x, int lane, int m, uint32_t lo_mask) {
  const uint32_t y = __shfl_xor_sync(0xffffffffu, x, m);
  const uint32_t hi_mask = lo_mask << m;
  return (lane & m) ? ((x & hi_mask) | ((y & hi_mask) >> m)) : ((x & lo_mask) | ((y & lo_mask) << m));
}

// Backward: the keep bits of key `key` for the `ncols` (16, 32 or 64)
// queries q0 .. q0 + ncols - 1, bit c <-> query q0 + c (x: 0-31, y: 32-63).
// One generator call covers 16 keys of one query, so lanes 16h .. 16h+15
// (keys key & ~15 .. +15) each draw the call of one query and a 16 x 16 bit
// transpose across the half-warp hands each lane the bits of its own key
// (key & 15 == lane & 15).  Every lane of the warp must call it with the
// same q0 and ncols.
template <typename Drop>
__device__ __forceinline__ uint2 key_keep_words(int key, int q0, int ncols, int lane, int bh, const Drop& drop) {
  const uint32_t kgrp = (uint32_t)(key >> 4);
  const int r16 = lane & 15;
  const uint32_t tt = drop.t * 0x01010101u;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int sc = 0; sc < 4; ++sc) {  // 16 queries per step
    if (16 * sc >= ncols) break;
    const uint4 g = philox4x32_10(make_uint4(kgrp, (uint32_t)(q0 + 16 * sc + r16), (uint32_t)bh, drop.offset),
                                  drop.k0, drop.k1);
    uint32_t x = keep_bits16(g, tt);  // row: query q0 + 16 sc + r16; bit k: key 16 kgrp + k
    x = transpose_step(x, lane, 8, 0x00FFu);
    x = transpose_step(x, lane, 4, 0x0F0Fu);
    x = transpose_step(x, lane, 2, 0x3333u);
    x = transpose_step(x, lane, 1, 0x5555u);
    w[sc >> 1] |= x << (16 * (sc & 1));
  }
  return make_uint2(w[0], w[1]);
}

}  // namespace fa

// Forward pass of exact attention on sm_103a: the kernel template, shared by
// the translation units that instantiate it (fa_fwd.cu: block-sparse;
// fa_fwd_dropout.cu: dropout; fa_fwd_varlen.cu: packed variable-length
// batches), and the helpers that fa_fwd_persist.cu (plain dense attention)
// and fa_fwd256.cu (d = 256) reuse.
//
// Algorithm: the online-softmax recurrence of "FlashAttention 为什么不需要存下
// 注意力矩阵" (jefxiong.cn), section 3.2 -- per query row a reference max m, a
// denominator l and an unnormalised accumulator O; a new key tile with
// larger scores rescales l and O by exp(m_old - m_new); the output is O / l
// and the saved statistic is LSE = m + ln l.  The loop order is queries
// outer, keys inner (the order the same page's section 05 attributes to
// FlashAttention-2), so O never leaves the chip until the end.
//
// Mapping onto one CTA (384 threads, one CTA per SM):
//   warp 0      TMA producer: Q tiles once, then K_j, V_j through a ring of
//               shared-memory slots (128-byte swizzle, 64-column slabs).
//   warp 1      allocates 512 TMEM columns; lane 0 issues every tcgen05.mma:
//               S_t = Q_t K_j^T (fp32 in TMEM) and O_t += P_t V_j with P_t
//               read from TMEM.
//   warps 4-7   softmax for query tile 0 (rows q0 .. q0+127),
//   warps 8-11  softmax for query tile 1 (rows q0+128 .. q0+255): each
//               thread owns one row (one TMEM lane), reads the 128 scores
//               of its row, updates m and l in the log2 domain with ex2,
//               writes P as packed 16-bit pairs over the S columns, and
//               rescales its O row in TMEM when needed.  The two tiles
//               ping-pong: while one softmax runs, the tensor core works
//               on the other tile.  At the end the same warps normalise O
//               and write their rows of O and LSE.
//
// Rescaling is lazy: the reference max of a row only moves when the new
// row max exceeds it by more than 8 (log2 units, i.e. a factor 256).  O and
// l always share one reference, so O / l and m + ln l are unchanged (the
// invariant of section 3.2 holds for any common reference; the max only
// prevents overflow, and 2^8 keeps every P below 256).  Two sums are kept:
// l over P in fp32 (for LSE) and l_mma over P as rounded to 16 bit for the
// PV product (for normalising O).
//
// Causal: key tiles entirely above the diagonal are never loaded or
// multiplied (section 4.5's whole-block skip); the diagonal tile and the
// ragged tail (keys >= N) are masked elementwise to -inf.  With Nq != Nk the
// diagonal is bottom-right aligned (query i sits at position i + Nk - Nq); a
// row that sees no key gets O = 0 and LSE = -inf.  Packed variable-length
// batches (SeqLayout) give every CTA its own sequence lengths and row bases.
// Block-sparse (SPARSE): the same skip driven by a mask of 128 x 128 blocks
// (section 06 generalises the whole-block skip to any pattern); a query tile
// that keeps no key tile writes O = 0 and LSE = -inf.
// Dropout (DROP): the softmax warps draw each entry's keep bit from the
// Philox generator (fa_philox.cuh) and zero the dropped P entries before
// they reach the PV product; l and LSE use the undropped P, and O is
// multiplied by the keep scale 1 / (1 - t / 256) in the epilogue.
#pragma once

#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "fa_layout.cuh"
#include "fa_philox.cuh"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;  // query rows per tile (tcgen05 M)
  static constexpr int BN = 128;  // keys per tile (tcgen05 N of S)
  static constexpr int QT = 2;    // query tiles per CTA
  static constexpr int SLAB = 128 * 64 * 2;  // 128 rows x 64 columns x 16 bit
  static constexpr int SLABS = D / 64;
  static constexpr int TILE = SLABS * SLAB;  // one 128 x D tile
  static constexpr int NS = D == 128 ? 4 : 8;  // K/V ring slots (5 at d = 128 measured 0.8% slower)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = QT * TILE;
  static constexpr int OFF_BAR = OFF_RING + NS * TILE;
  // q_full, ring_full[NS], ring_empty[NS], s_full[2], p_full[2], o_full[2], drain[2]
  static constexpr int NBAR = 1 + 2 * NS + 2 + 2 + 2 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;  // S0 | S1 | O0 | O1
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_O = 256;
};

__device__ __forceinline__ void unpack2(uint32_t v, bool bf16, float& lo, float& hi) {
  if (bf16) {
    lo = __uint_as_float(v << 16);
    hi = __uint_as_float(v & 0xffff0000u);
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&v);
    float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Bounded wait whose result is the same on every lane of the warp, so that
// warp-collective tcgen05 instructions after it are never split.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status) {
  const bool ok = mbar_wait(bar, parity, abort, status, kStatusTimeout);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait used only on the abort path: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

// One key tile of the online softmax for the calling thread's query row
// (one TMEM lane): reads the tile's 128 scores (columns tS ..), masks keys
// >= Nk and, when CAUSAL, keys > row_off (the tile's first row sees keys up
// to tile_off); moves the reference max m_ref when the tile's max exceeds it
// by more than kRescaleThreshold, scaling l, l_mma and, if `o_live` (earlier
// tiles of this row are in O), the O row in TMEM (columns tO ..); writes P
// as packed 16-bit pairs over the scores, with dropped entries zeroed when
// DROP.  sum2 / sumr2 return the tile's sum of P as computed and as rounded
// to 16 bit (pairs of partial sums), for the caller to add into l / l_mma
// after it has handed P to the tensor core.  The TMEM stores are not yet
// waited for.
template <int D, bool CAUSAL, bool BF16, bool DROP>
__device__ __forceinline__ void softmax_tile(uint32_t tS, uint32_t tO, int kbase, int Nk, int row_off,
                                             int tile_off, float scale_log2, bool o_live,
                                             const uint32_t (&keep)[4], float& m_ref, float& l, float& l_mma,
                                             uint64_t& sum2, uint64_t& sumr2) {
  constexpr int kBN = 128;
  float s[4][32];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + 32 * cc, s[cc]);
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(s[cc]);

  const bool need_mask = (kbase + kBN > Nk) || (CAUSAL && kbase + kBN - 1 > tile_off);
  if (need_mask) {
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int key = kbase + 32 * cc + i;
        if (key >= Nk || (CAUSAL && key > row_off)) s[cc][i] = neg_inf();
      }
  }
  float mx = s[0][0];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
#pragma unroll
    for (int i = 0; i < 32; i += 2) mx = max3(mx, s[cc][i], s[cc][i + 1]);
  const float m_new = fmaxf(m_ref, mx * scale_log2);
  float corr = 1.f;
  bool rescale_o = false;
  if (__any_sync(0xffffffffu, m_new > m_ref + kRescaleThreshold)) {
    const float m_use = (m_new == neg_inf()) ? 0.f : m_new;
    corr = ex2_approx(m_ref - m_use);
    l *= corr;
    l_mma *= corr;
    rescale_o = o_live;
    m_ref = m_use;
  }
  const float neg_m = (m_ref == neg_inf()) ? 0.f : -m_ref;
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
  const uint64_t nm2 = f2_pack(neg_m, neg_m);
  sum2 = f2_pack(0.f, 0.f);
  sumr2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {  // 32 scores -> 16 packed pairs -> 16 TMEM columns
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(s[cc][2 * i], s[cc][2 * i + 1]), sc2, nm2), x0, x1);
      const float p0 = ex2_approx(x0);
      const float p1 = ex2_approx(x1);
      sum2 = f2_add(sum2, f2_pack(p0, p1));
      pk[i] = pack2(p0, p1, BF16);
      float r0, r1;
      unpack2(pk[i], BF16, r0, r1);
      sumr2 = f2_add(sumr2, f2_pack(r0, r1));
    }
    if (DROP) {
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] &= pair_keep_mask(keep[cc], i);
    }
    tmem_st16(tS + 16 * cc, pk);
  }
  if (rescale_o) {
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
      float o[32];
      tmem_ld32(tO + 32 * cc, o);
      tmem_ld_wait(o);
      const uint64_t corr2 = f2_pack(corr, corr);
      uint32_t ou[32];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float a, b;
        f2_unpack(f2_mul(f2_pack(o[i], o[i + 1]), corr2), a, b);
        ou[i] = __float_as_uint(a);
        ou[i + 1] = __float_as_uint(b);
      }
      tmem_st32(tO + 32 * cc, ou);
    }
  }
}

// Epilogue of one query row: reads the row's O accumulator (columns tO ..),
// multiplies it by inv_l and, if `in_range`, writes the first dh features
// as 16-bit values to `orow` (dh / 8 16-byte chunks, contiguous in memory;
// features past dh, zero-padded inputs, are not stored).
template <int D, bool BF16>
__device__ __forceinline__ void store_o_row(uint32_t tO, uint4* orow, int dh, float inv_l, bool in_range) {
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    if (32 * cc >= dh) break;
    float ov[32];
    tmem_ld32(tO + 32 * cc, ov);
    tmem_ld_wait(ov);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack2(ov[2 * i] * inv_l, ov[2 * i + 1] * inv_l, BF16);
    if (in_range) {
#pragma unroll
      for (int q = 0; q < 4; ++q) orow[4 * cc + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
}

template <int D, bool CAUSAL, bool BF16, bool SPARSE, bool DROP, bool VARLEN>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  void* __restrict__ o,
                  float* __restrict__ lse, SeqLayout lay, int BH, int n_qblocks, float scale_log2,
                  const uint8_t* __restrict__ block_mask, int mask_heads, DropParams drop, int group,
                  unsigned int* status) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sRing = smem + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* ring_full = bars + 1;
  uint64_t* ring_empty = ring_full + C::NS;
  uint64_t* s_full = ring_empty + C::NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* drain = o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heads in groups of `group` (a group's K and V fit in about half of L2);
  // inside a group the heaviest work first: under the causal mask the last
  // query blocks see the most keys.
  const int gi = blockIdx.x / (group * n_qblocks);
  const int heads = min(group, BH - gi * group);  // the last group may be smaller
  const int within = blockIdx.x - gi * group * n_qblocks;
  const int bh = gi * group + within % heads;
  const int qb = n_qblocks - 1 - within / heads;
  const int q0 = qb * (C::QT * C::BM);
  const SeqView sv = seq_view<VARLEN>(lay, bh);
  if (!sv.ok && q0 == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadSeqlens);
  if (q0 >= sv.nq) return;  // past the end of a shorter (or rejected) sequence: the whole CTA leaves
  const int Nq = sv.nq, Nk = sv.nk;
  const int off = Nk - Nq;  // causal: key visible iff key <= row + off
  const int dh = lay.dh;
  const int n_kv = (Nk + C::BN - 1) / C::BN;
  // key tiles seen by query tile 0, and by query tile 1 (n1 >= n0)
  const int n0 = CAUSAL ? causal_key_tiles(q0 + C::BM - 1, off, n_kv, C::BN) : n_kv;
  const int n1 = CAUSAL ? causal_key_tiles(q0 + 2 * C::BM - 1, off, n_kv, C::BN) : n_kv;
  // Block-sparse: one mask byte per (128-row query tile, 128-key tile); a key
  // tile is loaded only if one of the two query tiles keeps it.
  const uint8_t* mrow0 = nullptr;
  const uint8_t* mrow1 = nullptr;
  bool t1_rows = true;  // query tile 1 starts inside the sequence
  if (SPARSE) {
    const uint8_t* mh = block_mask + (long long)(mask_heads == 1 ? 0 : bh) * n_kv * n_kv;
    const int qt0 = q0 / C::BM;
    t1_rows = qt0 + 1 < n_kv;
    mrow0 = mh + (long long)qt0 * n_kv;
    mrow1 = mh + (long long)(t1_rows ? qt0 + 1 : qt0) * n_kv;
  }
  auto act0 = [&](int j) { return j < n0 && (!SPARSE || mrow0[j] != 0); };
  auto act1 = [&](int j) { return !SPARSE || (t1_rows && mrow1[j] != 0); };  // j < n1 in every loop

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&o_full[t], 1);
      mbar_init(&drain[t], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto kslot = [](int j) { return (2 * j) % C::NS; };
  auto kpar = [](int j) { return (uint32_t)(((2 * j) / C::NS) & 1); };
  auto vslot = [](int j) { return (2 * j + 1) % C::NS; };
  auto vpar = [](int j) { return (uint32_t)(((2 * j + 1) / C::NS) & 1); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;  // K/V tiles whose copy has been started
      mbar_arrive_expect_tx(q_full, C::QT * C::TILE);
      for (int t = 0; t < C::QT; ++t) {
        const int2 c = sv.qcoord(q0 + t * C::BM);
        for (int s = 0; s < C::SLABS; ++s) tma_load_3d(sQ + t * C::TILE + s * C::SLAB, &tm_q, q_full, s * 64, c.x, c.y);
      }
      if constexpr (!SPARSE) {
        for (int u = 0; u < 2 * n1; ++u) {  // K_0, V_0, K_1, V_1, ...
          const int slot = u % C::NS;
          const uint32_t use = (uint32_t)(u / C::NS);
          if (!mbar_wait(&ring_empty[slot], (use & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
          mbar_arrive_expect_tx(&ring_full[slot], C::TILE);
          const CUtensorMap* m = (u & 1) ? &tm_v : &tm_k;
          const int2 c = sv.kcoord((u >> 1) * C::BN);
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(sRing + slot * C::TILE + s * C::SLAB, m, &ring_full[slot], s * 64, c.x, c.y);
          issued = u + 1;
        }
      } else {
        bool ok = true;
        for (int j = 0, u = 0; ok && j < n1; ++j) {  // u: position of key tile j in the load order
          if (SPARSE && !act0(j) && !act1(j)) continue;
          for (int kv = 0; kv < 2; ++kv) {
            const int uu = 2 * u + kv;
            const int slot = uu % C::NS;
            const uint32_t use = (uint32_t)(uu / C::NS);
            if (!(ok = mbar_wait(&ring_empty[slot], (use & 1) ^ 1, abort_flag, status, kStatusTimeout))) break;
            mbar_arrive_expect_tx(&ring_full[slot], C::TILE);
            const CUtensorMap* m = kv ? &tm_v : &tm_k;
            const int2 c = sv.kcoord(j * C::BN);
            for (int s = 0; s < C::SLABS; ++s)
              tma_load_3d(sRing + slot * C::TILE + s * C::SLAB, m, &ring_full[slot], s * 64, c.x, c.y);
            issued = uu + 1;
          }
          ++u;
        }
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        drain_wait(q_full, 0);
        for (int u = issued - C::NS < 0 ? 0 : issued - C::NS; u < issued; ++u)
          drain_wait(&ring_full[u % C::NS], (uint32_t)((u / C::NS) & 1));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, C::BN, BF16, false, false);
      constexpr uint32_t kIdPV = idesc_f16(128, D, BF16, false, true);
      const uint32_t sq = smem_u32(sQ);
      const uint32_t sring = smem_u32(sRing);
      // descriptors of the first Q tile and of ring slot 0 (K: K-major; V: MN-major)
      const uint64_t dq0 = sdesc_sw128(sq, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sring, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sring, C::SLAB, 1024);
      auto issue_s = [&](int t, int j) {
        const uint64_t da = sdesc_advance(dq0, t * C::TILE);
        const uint64_t db = sdesc_advance(dk0, kslot(j) * C::TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::SLAB + (kk & 3) * 32;
          mma_ss(tmem + C::COL_S + t * C::BN, sdesc_advance(da, off), sdesc_advance(db, off), kIdS, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int j, bool first) {
        const uint64_t dv = sdesc_advance(dv0, vslot(j) * C::TILE);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          mma_ts(tmem + C::COL_O + t * D, tmem + C::COL_S + t * C::BN + kk * 8,
                 sdesc_advance(dv, kk * 2048), kIdPV, (!first || kk > 0));
        }
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, status, kStatusTimeout);
      if constexpr (!SPARSE) {
        // Per key tile j: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j).  PV_t(j-1) is
        // issued before S_t(j), whose columns hold P_t(j-1), by the same
        // thread (in-order).  One thread issues both query tiles' products:
        // that order makes the tensor core alternate between the tiles while
        // each tile's softmax runs (two issuers, one per tile, measured
        // slower: 1.065 against 0.903 ms on the causal N = 8192, d = 128
        // forward).
        for (int j = 0; ok && j < n1; ++j) {
          if (!(ok = mbar_wait(&ring_full[kslot(j)], kpar(j), abort_flag, status, kStatusTimeout))) break;
          if (j >= 1 && !(ok = mbar_wait(&ring_full[vslot(j - 1)], vpar(j - 1), abort_flag, status, kStatusTimeout)))
            break;
          tc_fence_after();
          if (j >= 1 && j - 1 < n0) {
            if (!(ok = mbar_wait(&p_full[0], (j - 1) & 1, abort_flag, status, kStatusTimeout))) break;
            tc_fence_after();
            issue_pv(0, j - 1, j == 1);
            if (j == n0) mma_commit(&o_full[0]);  // query tile 0's last product (causal)
          }
          if (j < n0) {
            issue_s(0, j);
            mma_commit(&s_full[0]);
          }
          if (j >= 1) {
            if (!(ok = mbar_wait(&p_full[1], (j - 1) & 1, abort_flag, status, kStatusTimeout))) break;
            tc_fence_after();
            issue_pv(1, j - 1, j == 1);
            mma_commit(&ring_empty[vslot(j - 1)]);
          }
          issue_s(1, j);
          mma_commit(&s_full[1]);
          mma_commit(&ring_empty[kslot(j)]);
        }
        if (ok && n1 > 0) {
          const int jl = n1 - 1;
          ok = mbar_wait(&ring_full[vslot(jl)], vpar(jl), abort_flag, status, kStatusTimeout);
          tc_fence_after();
          if (ok && jl < n0) {
            ok = mbar_wait(&p_full[0], jl & 1, abort_flag, status, kStatusTimeout);
            tc_fence_after();
            if (ok) issue_pv(0, jl, jl == 0);
          }
          if (ok) {
            ok = mbar_wait(&p_full[1], jl & 1, abort_flag, status, kStatusTimeout);
            tc_fence_after();
            if (ok) issue_pv(1, jl, jl == 0);
          }
        }
        if (ok) {
          if (n0 == n1 || n0 == 0) mma_commit(&o_full[0]);
          mma_commit(&o_full[1]);
        }
        // Both query tiles run every key tile they see, query tile 1 also when
        // it starts past the last row (an odd number of query tiles): its
        // scores are computed and its rows never stored.
        if (ok) count_score_blocks(status, kCountForward, 4ull * (unsigned)(n0 + n1));
        if (!ok) {  // every MMA issued so far must finish before TMEM is freed
          mma_commit(&drain[0]);
          drain_wait(&drain[0], 0);
        }
      } else {
        // Per load-order position u: PV_0(prev), S_0(u), PV_1(prev), S_1(u), where
        // prev is the previous position; a query tile skips the products of the
        // key tiles it does not keep.  PV_t(prev) is issued before S_t(u), whose
        // columns hold P_t(prev), by the same thread (in-order).
        int prev = -1, c0 = 0, c1 = 0;  // previous position; S products issued per tile
        bool pa0 = false, pa1 = false;  // tile t kept the key tile at prev
        for (int j = 0, u = 0; ok && j < n1; ++j) {
          const bool a0 = act0(j), a1 = act1(j);
          if (SPARSE && !a0 && !a1) continue;
          if (prev >= 0 && !(ok = mbar_wait(&ring_full[vslot(prev)], vpar(prev), abort_flag, status, kStatusTimeout)))
            break;
          if (pa0) {
            if (!(ok = mbar_wait(&p_full[0], (c0 - 1) & 1, abort_flag, status, kStatusTimeout))) break;
            tc_fence_after();
            issue_pv(0, prev, c0 == 1);
          }
          if (!(ok = mbar_wait(&ring_full[kslot(u)], kpar(u), abort_flag, status, kStatusTimeout))) break;
          tc_fence_after();
          if (a0) {
            issue_s(0, u);
            mma_commit(&s_full[0]);
            ++c0;
          }
          if (pa1) {
            if (!(ok = mbar_wait(&p_full[1], (c1 - 1) & 1, abort_flag, status, kStatusTimeout))) break;
            tc_fence_after();
            issue_pv(1, prev, c1 == 1);
          }
          if (prev >= 0) mma_commit(&ring_empty[vslot(prev)]);
          if (a1) {
            issue_s(1, u);
            mma_commit(&s_full[1]);
            ++c1;
          }
          mma_commit(&ring_empty[kslot(u)]);
          prev = u;
          pa0 = a0;
          pa1 = a1;
          ++u;
        }
        if (ok && prev >= 0) {
          ok = mbar_wait(&ring_full[vslot(prev)], vpar(prev), abort_flag, status, kStatusTimeout);
          tc_fence_after();
          if (ok && pa0) {
            ok = mbar_wait(&p_full[0], (c0 - 1) & 1, abort_flag, status, kStatusTimeout);
            tc_fence_after();
            if (ok) issue_pv(0, prev, c0 == 1);
          }
          if (ok && pa1) {
            ok = mbar_wait(&p_full[1], (c1 - 1) & 1, abort_flag, status, kStatusTimeout);
            tc_fence_after();
            if (ok) issue_pv(1, prev, c1 == 1);
          }
        }
        if (ok) count_score_blocks(status, kCountForward, 4ull * (unsigned)(c0 + c1));
        if (ok) {
          mma_commit(&o_full[0]);
          mma_commit(&o_full[1]);
        }
        if (!ok) {  // every MMA issued so far must finish before TMEM is freed
          mma_commit(&drain[0]);
          drain_wait(&drain[0], 0);
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp >> 2) - 1;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
    const int row = q0 + t * C::BM + r;
    const int row_off = row + off;              // causal: key visible iff key <= row_off
    const int tile_off = q0 + t * C::BM + off;  // ... for the tile's first row
    const int n_t = t == 0 ? n0 : n1;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = lane_base + C::COL_S + t * C::BN;
    const uint32_t tO = lane_base + C::COL_O + t * D;

    float m_ref = neg_inf();  // reference max, log2 units of the scaled scores
    float l = 0.f;            // sum of exp2(score - m_ref): gives LSE
    float l_mma = 0.f;        // the same sum over P rounded to 16 bit: normalises O
    bool ok = true;
    int c = 0;  // key tiles processed so far by this query tile
    // Dropout keep bits of the next key tile (tiles are visited in order
    // 0, 1, ... when DROP): drawn while the tensor core works, so that the
    // generator stays off the path from S to P.
    uint32_t keep[4] = {0u, 0u, 0u, 0u};
    if (DROP && n_t > 0) tile_keep_bits<4>(keep, 0, row, bh, drop.offset, drop.k0, drop.k1, drop.t);
    for (int j = 0; j < n_t; ++j) {
      if constexpr (SPARSE) {
        if (!(t == 0 ? act0(j) : act1(j))) continue;
      } else {
        c = j;
      }
      if (!(ok = warp_wait(&s_full[t], c & 1, abort_flag, status))) break;
      tc_fence_after();
      uint64_t sum2, sumr2;  // this tile's sum of P as computed (fp32) and as rounded for the MMA
      softmax_tile<D, CAUSAL, BF16, DROP>(tS, tO, j * C::BN, Nk, row_off, tile_off, scale_log2, c > 0, keep, m_ref,
                                          l, l_mma, sum2, sumr2);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
      if (DROP && j + 1 < n_t) tile_keep_bits<4>(keep, (j + 1) * C::BN, row, bh, drop.offset, drop.k0, drop.k1, drop.t);
      float a, b;
      f2_unpack(sum2, a, b);
      l += a + b;
      f2_unpack(sumr2, a, b);
      l_mma += a + b;
      ++c;
    }

    // ------------------------------------------------------------ epilogue
    // Block-sparse and dropout instances (dense layouts) stage O in shared
    // memory and store it with TMA; the plain dense instances measured
    // faster with per-row stores, and packed layouts need them (a tile's
    // last rows can belong to the next sequence).
    constexpr bool kStageO = !VARLEN && (SPARSE || DROP);
    if (ok) ok = warp_wait(&o_full[t], 0, abort_flag, status);
    const long long frow = sv.qflat(row);
    const bool has_o = ok && c > 0;
    if (ok && c == 0) {  // no key tile for this query tile: empty softmax, O = 0, LSE = -inf
      uint4* orow = reinterpret_cast<uint4*>(o) + frow * (dh / 8);
      if (row < Nq) {
        for (int q = 0; q < dh / 8; ++q) orow[q] = make_uint4(0u, 0u, 0u, 0u);
        lse[frow] = neg_inf();
      }
    } else if (has_o) {
      tc_fence_after();
      // O is divided by the sum of the rounded weights that entered the MMA,
      // so each output row stays a convex combination of V rows; the
      // rounding of the dominant weight then cancels instead of showing up
      // at the 16-bit resolution of P.
      // A row that saw no key (bottom-right causal with Nq > Nk) has l = 0 and
      // O = 0 in TMEM: it stays 0, and its LSE is -inf.
      const float inv_l = l_mma > 0.f ? (DROP ? drop.keep_scale : 1.f) / l_mma : 0.f;
      if constexpr (kStageO) {
        // The warpgroup stages its 128 x D tile of O in the (now unused)
        // shared-memory tile of Q_t, in the 128-byte-swizzled slabs the O
        // tensor map describes; one thread stores it with TMA below.
        uint8_t* stage = sQ + t * C::TILE;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          float ov[32];
          tmem_ld32(tO + 32 * cc, ov);
          tmem_ld_wait(ov);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack2(ov[2 * i] * inv_l, ov[2 * i + 1] * inv_l, BF16);
          uint8_t* slab = stage + ((32 * cc) >> 6) * C::SLAB;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(slab + sw128_offset(r, (32 * cc & 63) + 8 * q)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      } else {
        store_o_row<D, BF16>(tO, reinterpret_cast<uint4*>(o) + frow * (dh / 8), dh, inv_l, row < Nq);
      }
      if (row < Nq) {
        const float m_fin = (m_ref == neg_inf()) ? 0.f : m_ref;
        lse[frow] = (m_fin + __log2f(l)) * kLn2;
      }
    }
    if constexpr (kStageO) {
      // Every warp of the warpgroup reaches this barrier once, whatever its
      // path above; rows past Nq and features past dh fall outside the O map
      // and are not written.
      fence_async_smem();
      named_barrier_sync(1 + t, 128);
      const int row0 = q0 + t * C::BM;
      if (r == 0 && has_o && row0 < Nq && !*abort_flag) {
        const int2 cq = sv.qcoord(row0);
#pragma unroll
        for (int sl = 0; sl < C::SLABS; ++sl)
          if (64 * sl < dh) tma_store_3d(&tm_o, sQ + t * C::TILE + sl * C::SLAB, 64 * sl, cq.x, cq.y);
        tma_store_commit();
        tma_store_wait_read();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL, bool BF16, bool SPARSE, bool DROP, bool VARLEN>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fa_fwd_kernel<D, CAUSAL, BF16, SPARSE, DROP, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qblocks = (a.lay.Nq + C::QT * C::BM - 1) / (C::QT * C::BM);
  const long long grid = (long long)n_qblocks * a.BH;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // K and V of a head take 4 * Nk * D bytes; a group keeps them within ~64 MB of L2.
  const long long per_head = 4LL * a.lay.Nk * D;
  const int group = (int)std::max(1LL, std::min(64LL, (64LL << 20) / (per_head > 0 ? per_head : 1)));
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.o, a.lse, a.lay, a.BH,
                                                         n_qblocks,
                                                         a.scale_log2, a.block_mask, a.mask_heads, a.drop, group,
                                                         a.status);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fa

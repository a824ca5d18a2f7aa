// Forward pass, dense layouts without block mask or dropout.
//
// The arithmetic is that of the kernel in fa_fwd_kernel.cuh (the online-
// softmax recurrence of "FlashAttention 为什么不需要存下注意力矩阵", section
// 3.2, queries outer and keys inner; causal whole-tile skip of section 4.5,
// the same softmax_tile and store_o_row), and the two produce bitwise equal
// O and LSE.  What differs is how work and data reach the tensor core:
//   - Q has a producer warp of its own and full / empty barriers per query
//     tile, so the K / V producer never waits for Q;
//   - O_t has its own full / empty barriers per query tile: softmax
//     warpgroup 0 (one key tile fewer under the causal mask) writes its O
//     rows while warpgroup 1 finishes the item;
//   - at d = 64, and at d = 128 with short keys, CTAs are persistent: the grid has one CTA per
//     work item (a head and 256 query rows, heads in L2 groups, heaviest
//     query blocks first), but a running CTA, a few key tiles before the end
//     of its item, cancels through cluster launch control the launch of a
//     CTA that has not started and does that CTA's item itself.  TMEM,
//     barriers and descriptors are then set up once per SM, the K / V ring
//     flows on into the next item, and the next item's Q is pulled into L2
//     and loaded while the current item ends.  At d = 128 with long keys
//     one CTA per item measured faster (the cancellation answers come back
//     only roughly in grid order, and the chained items' running phase bases
//     cost the single MMA-issuing thread instructions, which items of many
//     key tiles do not win back).
// The MMA issuer's loop per item is the one-shot kernel's: PV_0(j-1), S_0(j),
// PV_1(j-1), S_1(j) from one thread.
//
// Roles (384 threads, one CTA per SM):
//   warp 0      K / V producer (TMA through the ring of shared-memory slots)
//               and, when persistent, the one that asks for the next item
//   warp 1      TMEM allocation; lane 0 issues every tcgen05.mma
//   warp 2      Q producer (and L2 prefetch of the next item's Q)
//   warps 4-11  softmax and epilogue for query tiles 0 and 1 (one row per
//               thread)
// When persistent, the answer for "the item after item k" (k counts this
// CTA's items) sits in slot k % 2 and is read by every role before the slot
// is reused.
#include "fa_fwd_kernel.cuh"

namespace fa {
namespace {

template <int D>
struct PersistCfg {
  using F = FwdCfg<D>;
  static constexpr int BM = F::BM, BN = F::BN, QT = F::QT;
  static constexpr int SLAB = F::SLAB, SLABS = F::SLABS, TILE = F::TILE;
  static constexpr int NS = F::NS;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = QT * TILE;
  static constexpr int OFF_BAR = OFF_RING + NS * TILE;
  // q_full[2], q_empty[2], ring_full[NS], ring_empty[NS], s_full[2], p_full[2],
  // o_full[2], o_empty[2], next_full[2], next_empty[2], drain
  static constexpr int NBAR = 2 + 2 + 2 * NS + 2 + 2 + 2 + 2 + 2 + 2 + 1;
  static constexpr int OFF_NEXT = (OFF_BAR + NBAR * 8 + 15) & ~15;  // two 16-byte answers
  static constexpr int OFF_MISC = OFF_NEXT + 32;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;  // S0 | S1 | O0 | O1
  static constexpr uint32_t COL_S = F::COL_S;
  static constexpr uint32_t COL_O = F::COL_O;
  // Readers of each answer besides the K / V producer that asks: the Q
  // producer, the MMA issuer, 8 softmax warps.
  static constexpr uint32_t NEXT_READERS = 10;
};

// Whether CTAs take further items, measured with the same code otherwise: at
// d = 64 a CTA that stays resident was 2-4% faster than one CTA per item (N =
// 4096); at d = 128 causal it is faster for short keys (N = 1024: 9%, 2048:
// 3.6%) and slower for long ones (4096: 1%, 8192: 4%), where items are long
// enough to amortise their start and the claimed items' order costs more.
template <int D>
constexpr bool kAlwaysPersistent = D == 64;
constexpr int kPersistMaxKeys = 2048;  // d = 128: persistent up to this many keys

// The K / V producer asks for the next item when it starts loading the
// kClaimAhead-th last key tile of the current one (it runs NS / 2 key tiles
// ahead of the tensor core).
constexpr int kClaimAhead = 2;

template <int D, bool CAUSAL, bool BF16, bool PERSIST>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o,
                          float* __restrict__ lse, SeqLayout lay, int BH, int n_qblocks, float scale_log2,
                          int group, unsigned int* status) {
  using C = PersistCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sRing = smem + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + 2;
  uint64_t* ring_full = q_empty + 2;
  uint64_t* ring_empty = ring_full + C::NS;
  uint64_t* s_full = ring_empty + C::NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* o_empty = o_full + 2;
  uint64_t* next_full = o_empty + 2;
  uint64_t* next_empty = next_full + 2;
  uint64_t* drain = next_empty + 2;
  uint8_t* next_ans = smem + C::OFF_NEXT;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int Nq = lay.Nq, Nk = lay.Nk;
  const int off = Nk - Nq;  // causal: key visible iff key <= row + off
  const int dh = lay.dh;
  const int n_kv = (Nk + C::BN - 1) / C::BN;

  // Work item w -> head and first query row: heads in groups of `group`
  // (a group's K and V fit in about half of L2), inside a group the
  // heaviest query blocks first (under the causal mask the last query
  // blocks see the most keys).
  auto item_bh = [&](int w) {
    const int gi = w / (group * n_qblocks);
    const int heads = min(group, BH - gi * group);  // the last group may be smaller
    return gi * group + (w - gi * group * n_qblocks) % heads;
  };
  auto item_q0 = [&](int w) {
    const int gi = w / (group * n_qblocks);
    const int heads = min(group, BH - gi * group);
    return (n_qblocks - 1 - (w - gi * group * n_qblocks) / heads) * (C::QT * C::BM);
  };
  // key tiles seen by query tile 0 and by query tile 1 (n1 >= n0)
  auto tiles0 = [&](int q0) { return CAUSAL ? causal_key_tiles(q0 + C::BM - 1, off, n_kv, C::BN) : n_kv; };
  auto tiles1 = [&](int q0) { return CAUSAL ? causal_key_tiles(q0 + 2 * C::BM - 1, off, n_kv, C::BN) : n_kv; };
  auto slot = [](uint32_t u) { return (int)(u % C::NS); };
  auto par = [](uint32_t u) { return (uint32_t)((u / C::NS) & 1); };

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_empty[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_full[t], 1);
      mbar_init(&o_empty[t], 4);
      mbar_init(&next_full[t], 1);
      mbar_init(&next_empty[t], C::NEXT_READERS);
    }
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    mbar_init(drain, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ K / V producer, scheduler
    if (lane == 0) {
      uint32_t u = 0;  // tiles whose copy has been started: K_0, V_0, K_1, V_1, ... over all items
      bool ok = true, asked = false;
      int k = 0;
      // Asks for the item after item k.  Its slot was last read after item k - 2.
      auto ask = [&]() -> bool {
        const int sl = k & 1;
        if (k >= 2 && !mbar_wait(&next_empty[sl], ((k - 2) >> 1) & 1, abort_flag, status, kStatusTimeout))
          return false;
        mbar_arrive_expect_tx(&next_full[sl], 16);
        clc_try_cancel(next_ans + 16 * sl, &next_full[sl]);
        asked = true;
        return true;
      };
      for (int w = blockIdx.x; ok; ++k) {
        const int bh = item_bh(w);
        const int n1 = tiles1(item_q0(w));
        // The next item is claimed only near the end of this one, so that
        // the CTA that finishes first takes the heaviest item left (a claim
        // at the start would pair heavy items with heavy ones).
        const int claim_at = PERSIST ? max(0, n1 - kClaimAhead) : -1;
        for (int j = 0; ok && j < n1; ++j) {
          if (j == claim_at && !(ok = ask())) break;
          for (int kv = 0; kv < 2; ++kv, ++u) {
            if (!(ok = mbar_wait(&ring_empty[slot(u)], par(u) ^ 1, abort_flag, status, kStatusTimeout))) break;
            mbar_arrive_expect_tx(&ring_full[slot(u)], C::TILE);
            const CUtensorMap* m = kv ? &tm_v : &tm_k;
            for (int s = 0; s < C::SLABS; ++s)
              tma_load_3d(sRing + slot(u) * C::TILE + s * C::SLAB, m, &ring_full[slot(u)], s * 64, j * C::BN, bh);
          }
        }
        if (!PERSIST) break;
        if (ok && n1 == 0) ok = ask();
        if (!ok || !(ok = mbar_wait(&next_full[k & 1], (k >> 1) & 1, abort_flag, status, kStatusTimeout))) break;
        asked = false;
        int nw;
        if (!clc_cancelled(next_ans + 16 * (k & 1), &nw)) break;
        w = nw;
      }
      if (*abort_flag) {  // let every copy and answer in flight land before the CTA exits
        for (uint32_t x = u > (uint32_t)C::NS ? u - C::NS : 0; x < u; ++x) drain_wait(&ring_full[slot(x)], par(x));
        if (asked) drain_wait(&next_full[k & 1], (k >> 1) & 1);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ Q producer
    if (lane == 0) {
      bool ok = true;
      int k = 0;
      int loaded[2] = {-1, -1};  // last item whose Q tile t was requested
      for (int w = blockIdx.x; ok; ++k) {
        const int bh = item_bh(w), q0 = item_q0(w);
        for (int t = 0; ok && t < C::QT; ++t) {
          if (k >= 1 && !(ok = mbar_wait(&q_empty[t], (k - 1) & 1, abort_flag, status, kStatusTimeout))) break;
          mbar_arrive_expect_tx(&q_full[t], C::TILE);
          for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(sQ + t * C::TILE + s * C::SLAB, &tm_q, &q_full[t], s * 64, q0 + t * C::BM, bh);
          loaded[t] = k;
        }
        if (!PERSIST) break;
        if (!ok || !(ok = mbar_wait(&next_full[k & 1], (k >> 1) & 1, abort_flag, status, kStatusTimeout))) break;
        int nw;
        const bool more = clc_cancelled(next_ans + 16 * (k & 1), &nw);
        mbar_arrive(&next_empty[k & 1]);
        if (!more) break;
        w = nw;
        // pull the next item's Q into L2 while this item's last products run
        const int nbh = item_bh(w), nq0 = item_q0(w);
        for (int t = 0; t < C::QT; ++t)
          if (nq0 + t * C::BM < Nq)
            for (int s = 0; s < C::SLABS; ++s) tma_prefetch_l2_3d(&tm_q, s * 64, nq0 + t * C::BM, nbh);
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        for (int t = 0; t < C::QT; ++t)
          if (loaded[t] >= 0) drain_wait(&q_full[t], loaded[t] & 1);
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
      // S_t = Q_t K^T with K at ring position u
      auto issue_s = [&](int t, uint32_t u) {
        const uint64_t da = sdesc_advance(dq0, t * C::TILE);
        const uint64_t db = sdesc_advance(dk0, slot(u) * C::TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * C::SLAB + (kk & 3) * 32;
          mma_ss(tmem + C::COL_S + t * C::BN, sdesc_advance(da, koff), sdesc_advance(db, koff), kIdS, kk > 0);
        }
      };
      // O_t (+)= P_t V with V at ring position u, P_t over the columns of S_t
      auto issue_pv = [&](int t, uint32_t u, bool accumulate) {
        const uint64_t dv = sdesc_advance(dv0, slot(u) * C::TILE);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          mma_ts(tmem + C::COL_O + t * D, tmem + C::COL_S + t * C::BN + kk * 8,
                 sdesc_advance(dv, kk * 2048), kIdPV, (accumulate || kk > 0));
        }
      };
      uint32_t u0 = 0;                // ring position of the item's K_0 (K_j at u0 + 2j, V_j at u0 + 2j + 1)
      uint32_t np0 = 0, np1 = 0;      // phases of p_full[0] / p_full[1] before the item
      unsigned long long blocks = 0;  // 64 x 64 score blocks computed
      bool ok = true;
      for (int k = 0, w = blockIdx.x; ok; ++k) {
        const int q0 = item_q0(w);
        const int n0 = tiles0(q0), n1 = tiles1(q0);
        blocks += 4ull * (unsigned)(n0 + n1);
        if (!(ok = mbar_wait(&q_full[0], k & 1, abort_flag, status, kStatusTimeout) &&
                   mbar_wait(&q_full[1], k & 1, abort_flag, status, kStatusTimeout)))
          break;
        // The item's first P V product of query tile t overwrites O_t: the
        // previous item's rows of O_t must have been read.
        auto o_free = [&](int t) {
          return k == 0 || mbar_wait(&o_empty[t], (k - 1) & 1, abort_flag, status, kStatusTimeout);
        };
        if (n0 == 0) mma_commit(&q_empty[0]);
        if (n1 == 0) mma_commit(&q_empty[1]);
        // Per key tile j: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j), as in the
        // one-shot kernel.
        for (int j = 0; ok && j < n1; ++j) {
          const uint32_t uk = u0 + 2 * j;
          if (!(ok = mbar_wait(&ring_full[slot(uk)], par(uk), abort_flag, status, kStatusTimeout))) break;
          if (j >= 1 && !(ok = mbar_wait(&ring_full[slot(uk - 1)], par(uk - 1), abort_flag, status, kStatusTimeout)))
            break;
          tc_fence_after();
          if (j >= 1 && j - 1 < n0) {
            if (!(ok = mbar_wait(&p_full[0], (np0 + j - 1) & 1, abort_flag, status, kStatusTimeout))) break;
            if (j == 1 && !(ok = o_free(0))) break;
            tc_fence_after();
            issue_pv(0, uk - 1, j > 1);
            if (j == n0) mma_commit(&o_full[0]);  // query tile 0's last product (causal)
          }
          if (j < n0) {
            issue_s(0, uk);
            mma_commit(&s_full[0]);
            if (j == n0 - 1) mma_commit(&q_empty[0]);
          }
          if (j >= 1) {
            if (!(ok = mbar_wait(&p_full[1], (np1 + j - 1) & 1, abort_flag, status, kStatusTimeout))) break;
            if (j == 1 && !(ok = o_free(1))) break;
            tc_fence_after();
            issue_pv(1, uk - 1, j > 1);
            mma_commit(&ring_empty[slot(uk - 1)]);
          }
          issue_s(1, uk);
          mma_commit(&s_full[1]);
          if (j == n1 - 1) mma_commit(&q_empty[1]);
          mma_commit(&ring_empty[slot(uk)]);
        }
        if (ok && n1 > 0) {
          const int jl = n1 - 1;
          const uint32_t uv = u0 + 2 * jl + 1;
          ok = mbar_wait(&ring_full[slot(uv)], par(uv), abort_flag, status, kStatusTimeout);
          tc_fence_after();
          if (ok && jl < n0) {
            ok = mbar_wait(&p_full[0], (np0 + jl) & 1, abort_flag, status, kStatusTimeout) && (jl > 0 || o_free(0));
            tc_fence_after();
            if (ok) issue_pv(0, uv, jl > 0);
          }
          if (ok) {
            ok = mbar_wait(&p_full[1], (np1 + jl) & 1, abort_flag, status, kStatusTimeout) && (jl > 0 || o_free(1));
            tc_fence_after();
            if (ok) {
              issue_pv(1, uv, jl > 0);
              mma_commit(&ring_empty[slot(uv)]);
            }
          }
        }
        if (!ok) break;
        // A query tile without key tiles ends its item here; o_full[t] may
        // run only one phase ahead of warpgroup t.
        if (n0 == n1 || n0 == 0) {
          if (n0 == 0 && !(ok = o_free(0))) break;
          mma_commit(&o_full[0]);
        }
        if (n1 == 0 && !(ok = o_free(1))) break;
        mma_commit(&o_full[1]);
        u0 += 2 * (uint32_t)n1;
        np0 += (uint32_t)n0;
        np1 += (uint32_t)n1;
        if (!PERSIST) break;
        if (!(ok = mbar_wait(&next_full[k & 1], (k >> 1) & 1, abort_flag, status, kStatusTimeout))) break;
        int nw;
        const bool more = clc_cancelled(next_ans + 16 * (k & 1), &nw);
        mbar_arrive(&next_empty[k & 1]);
        if (!more) break;
        w = nw;
      }
      if (ok) count_score_blocks(status, kCountForward, blocks);
      if (!ok) {  // every MMA issued so far must finish before TMEM is freed
        mma_commit(drain);
        drain_wait(drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax, epilogue
    const int t = (warp >> 2) - 1;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = lane_base + C::COL_S + t * C::BN;
    const uint32_t tO = lane_base + C::COL_O + t * D;
    const uint32_t no_drop[4] = {0u, 0u, 0u, 0u};
    uint32_t ns = 0;  // S tiles taken (phases of s_full)
    bool ok = true;
    for (int k = 0, w = blockIdx.x; ok; ++k) {
      const int bh = item_bh(w), q0 = item_q0(w);
      const int row = q0 + t * C::BM + r;
      const int row_off = row + off;              // causal: key visible iff key <= row_off
      const int tile_off = q0 + t * C::BM + off;  // ... for the tile's first row
      const int n_t = t == 0 ? tiles0(q0) : tiles1(q0);
      float m_ref = neg_inf();  // reference max, log2 units of the scaled scores
      float l = 0.f;            // sum of exp2(score - m_ref): gives LSE
      float l_mma = 0.f;        // the same sum over P rounded to 16 bit: normalises O
      for (int j = 0; j < n_t; ++j, ++ns) {
        if (!(ok = warp_wait(&s_full[t], ns & 1, abort_flag, status))) break;
        tc_fence_after();
        uint64_t sum2, sumr2;
        softmax_tile<D, CAUSAL, BF16, false>(tS, tO, j * C::BN, Nk, row_off, tile_off, scale_log2, j > 0, no_drop,
                                             m_ref, l, l_mma, sum2, sumr2);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[t]);
        float a, b;
        f2_unpack(sum2, a, b);
        l += a + b;
        f2_unpack(sumr2, a, b);
        l_mma += a + b;
      }
      if (!ok || !(ok = warp_wait(&o_full[t], k & 1, abort_flag, status))) break;
      tc_fence_after();
      const long long frow = (long long)bh * Nq + row;
      if (n_t == 0) {  // no key tile for this query tile: O = 0, LSE = -inf
        if (row < Nq) {
          uint4* orow = reinterpret_cast<uint4*>(o) + frow * (dh / 8);
          for (int q = 0; q < dh / 8; ++q) orow[q] = make_uint4(0u, 0u, 0u, 0u);
          lse[frow] = neg_inf();
        }
      } else {
        // O / l over the rounded weights (see the one-shot kernel); a row
        // that saw no key has l = 0, O = 0 and LSE = -inf.
        const float inv_l = l_mma > 0.f ? 1.f / l_mma : 0.f;
        store_o_row<D, BF16>(tO, reinterpret_cast<uint4*>(o) + frow * (dh / 8), dh, inv_l, row < Nq);
        if (row < Nq) {
          const float m_fin = (m_ref == neg_inf()) ? 0.f : m_ref;
          lse[frow] = (m_fin + __log2f(l)) * kLn2;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[t]);
      if (!PERSIST) break;
      if (!(ok = warp_wait(&next_full[k & 1], (k >> 1) & 1, abort_flag, status))) break;
      int nw;
      const bool more = clc_cancelled(next_ans + 16 * (k & 1), &nw);
      __syncwarp();
      if (lane == 0) mbar_arrive(&next_empty[k & 1]);
      if (!more) break;
      w = nw;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL, bool BF16, bool PERSIST>
cudaError_t launch_persist_k(const FwdArgs& a, cudaStream_t stream) {
  using C = PersistCfg<D>;
  auto kern = fa_fwd_persist_kernel<D, CAUSAL, BF16, PERSIST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qblocks = (a.lay.Nq + C::QT * C::BM - 1) / (C::QT * C::BM);
  const long long grid = (long long)n_qblocks * a.BH;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // K and V of a head take 4 * Nk * D bytes; a group keeps them within ~64 MB of L2.
  const long long per_head = 4LL * a.lay.Nk * D;
  const int group = (int)std::max(1LL, std::min(64LL, (64LL << 20) / (per_head > 0 ? per_head : 1)));
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, a.lay, a.BH, n_qblocks,
                                                         a.scale_log2, group, a.status);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_persist_t(const FwdArgs& a, cudaStream_t stream) {
  if constexpr (kAlwaysPersistent<D>) {
    return launch_persist_k<D, CAUSAL, BF16, true>(a, stream);
  } else {
    return a.lay.Nk <= kPersistMaxKeys ? launch_persist_k<D, CAUSAL, BF16, true>(a, stream)
                                       : launch_persist_k<D, CAUSAL, BF16, false>(a, stream);
  }
}

}  // namespace

cudaError_t launch_forward_persistent(int d, bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream) {
#define FA_PERSIST_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_persist_t<DD, CC, BB>(a, stream);
  FA_PERSIST_CASE(64, false, false)
  FA_PERSIST_CASE(64, false, true)
  FA_PERSIST_CASE(64, true, false)
  FA_PERSIST_CASE(64, true, true)
  FA_PERSIST_CASE(128, false, false)
  FA_PERSIST_CASE(128, false, true)
  FA_PERSIST_CASE(128, true, false)
  FA_PERSIST_CASE(128, true, true)
#undef FA_PERSIST_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa

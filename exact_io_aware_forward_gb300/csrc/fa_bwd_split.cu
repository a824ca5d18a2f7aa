// Backward pass with dQ in a kernel of its own (the "separate pass" strategy
// for dQ), on sm_103a: a dK / dV kernel over 128-query tiles and a dQ kernel
// over 128-key tiles.
//
// Math ("FlashAttention 为什么不需要存下注意力矩阵", jefxiong.cn, section 3.3):
// with P = exp(s Q K^T - LSE) recomputed tile by tile on chip and
// D_i = dO_i . O_i,
//   dP = dO V^T,  dS = P * (dP - D),  dV = P^T dO,  dK = s dS^T Q,  dQ = s dS K.
// Nothing N x N leaves the chip.  Both kernels recompute P and dP; the dQ
// kernel needs no float32 accumulator in device memory and no atomics, and
// the dK / dV kernel, free of the dQ product and its reductions, has the TMEM
// for 128-query tiles (every product N >= 128).
//
// fa_bwd_dkdv_split_kernel -- one CTA per 128-key tile (the MMA M dimension),
// looping over 128-query tiles.  TMEM (D = 128):
//   S^T 128 | dP^T 128 | dV 128 | dK 128   (D = 64: dV 64 | dK 64)
//   S^T = K Q_i^T, dP^T = V dO_i^T;  P^T goes to a shared-memory buffer (the
//   A operand of dV += P^T dO_i), so S^T(i+1) can be computed as soon as the
//   compute warps hold S^T(i) in registers; dS^T is written as 16-bit pairs
//   over the first half of each compute warpgroup's own dP^T columns, where
//   dK += dS^T Q_i reads it as a TMEM A operand.
// Warps (384 threads):
//   0      TMA: K, V once; Q_i, dO_i through a ring (2 stages at D = 128).
//   1      TMEM allocation; lane 0 issues S^T(i+1) and dV(i).
//   2      lane 0 issues dP^T(i+1) and dK(i).
//   4-7 / 8-11  compute warpgroup h = 0 / 1: one key row per thread (TMEM
//          lane), query columns [64h, 64h + 64): P^T from S^T and LSE (pass
//          1, P kept in registers), then dS^T from dP^T and D (pass 2).
//   dK(i) reads dS^T(i) from the dP^T columns before dP^T(i+1) overwrites
//   them (same issuing thread, in order).
//
// fa_bwd_dq_kernel -- one CTA per 128-query tile, looping over 128-key tiles.
// Q of the tile is copied once into TMEM as an A operand.  TMEM (D = 128):
//   Q 64 | S 128 | dP 128 | dQ 128 | dS 64
//   S = Q K_j^T (Q from TMEM), dP = dO V_j^T (dO from shared memory), dS
//   (16-bit pairs), dQ += dS K_j accumulates in TMEM for the whole key loop
//   and is scaled and stored once.
// Warps (384 threads): 0 TMA (Q, dO once; K_j through a 3-slot ring, V_j
//   through a 2-slot ring), 1 TMEM allocation and the issuer of S, 2 the
//   issuer of dP (dO from shared memory), 3 the issuer of dQ, 4-7 / 8-11
//   compute warpgroups, one query row per thread and key columns
//   [64h, 64h + 64).  dS has TMEM columns of its own, so dP(j+1) never waits
//   for dQ(j).
//
// Causal (square, top-left): query tiles entirely above the diagonal, and
// key tiles entirely right of it, are skipped by the loop bounds (the
// whole-block skip of section 4.5); the diagonal tile is masked elementwise.
// Dense [B, H, N, d] layouts, no block mask, no dropout; d = 96 runs the
// D = 128 instances (features 96-127 read as zero, never stored).
#include "fa_bwd_kernel.cuh"

namespace fa {
namespace {

template <int D>
struct SplitCfg {
  static constexpr int BKV = 128;                  // keys per tile
  static constexpr int BQ = 128;                   // queries per tile
  static constexpr int SLABS = D / 64;
  static constexpr int SLAB = 128 * 128;           // 128 rows x 64 columns x 16 bit
  static constexpr int TILE = SLABS * SLAB;        // one 128 x D tile
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
};

// ---------------------------------------------------------------- dK / dV
template <int D>
struct DkdvSplitCfg : SplitCfg<D> {
  using B = SplitCfg<D>;
  // Of the 8 pairs of exponentials in a 16-column chunk, this many are
  // evaluated on the FMA pipe (exp2_poly2), the rest on the special-function
  // unit.
  static constexpr int POLY_PAIRS = 0;
  static constexpr int CWG = 4;                    // compute warpgroups, 32 query columns each
  static constexpr int THREADS = 128 + 128 * CWG;
  static constexpr int QS = D == 128 ? 2 : 4;      // Q / dO stages
  static constexpr int PT_SLAB = 128 * 128;        // 128 keys x 64 queries x 16 bit
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = B::TILE;
  static constexpr int OFF_Q = 2 * B::TILE;        // [QS]
  static constexpr int OFF_DO = OFF_Q + QS * B::TILE;
  static constexpr int OFF_PT = OFF_DO + QS * B::TILE;  // P^T, 2 slabs (query halves), A operand of dV
  static constexpr int OFF_LD = OFF_PT + 2 * PT_SLAB;   // [CWG][-LSE log2e, -D][32] floats
  static constexpr int OFF_BAR = OFF_LD + CWG * 2 * 32 * 4;
  // kv_full, q_full[QS], q_empty[QS], s_full, s_empty, p_full, pt_empty, dp_full, ds_full, dkdv_done,
  // drain[2], ld_full[CWG], ld_empty[CWG]
  static constexpr int NBAR = 1 + 2 * QS + 7 + 2 + 2 * CWG;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = 128;
  static constexpr uint32_t COL_DV = 256;
  static constexpr uint32_t COL_DK = 256 + D;
  static_assert(COL_DK + D <= B::TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL, bool BF16, bool SPARSE, bool VARLEN, bool DROP>
__global__ void __launch_bounds__(DkdvSplitCfg<D>::THREADS, 1)
    fa_bwd_dkdv_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                             const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                             void* __restrict__ dk, void* __restrict__ dv, const float* __restrict__ lse,
                             const float* __restrict__ delta, SeqLayout lay, int BH, int dh, float scale,
                             float scale_log2, const uint8_t* __restrict__ block_mask, int mask_heads,
                             DropParams drop, int group, unsigned int* status) {
  using C = DkdvSplitCfg<D>;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sPT = smem + C::OFF_PT;
  float* sLD = reinterpret_cast<float*>(smem + C::OFF_LD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = kv_full + 1;
  uint64_t* q_empty = q_full + C::QS;
  uint64_t* s_full = q_empty + C::QS;
  uint64_t* s_empty = s_full + 1;    // every compute warp holds S^T(i) in registers
  uint64_t* p_full = s_empty + 1;    // P^T(i) written to shared memory
  uint64_t* pt_empty = p_full + 1;   // dV(i) has read P^T(i)
  uint64_t* dp_full = pt_empty + 1;
  uint64_t* ds_full = dp_full + 1;   // dS^T(i) written over dP^T(i) in TMEM
  uint64_t* dkdv_done = ds_full + 1;
  uint64_t* drain = dkdv_done + 1;   // [2]
  uint64_t* ld_full = drain + 2;     // [CWG]
  uint64_t* ld_empty = ld_full + C::CWG;  // [CWG]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heads in groups of `group` (a group's Q and dO fit in about half of L2);
  // inside a group key tile 0 of every head (which meets every query tile
  // under the causal mask) first, then key tile 1, ...
  const int n_kt = (lay.Nk + C::BKV - 1) / C::BKV;  // key tiles of the longest sequence
  const int gi = blockIdx.x / (group * n_kt);
  const int heads = min(group, BH - gi * group);
  const int within = blockIdx.x - gi * group * n_kt;
  const int bh = gi * group + within % heads;
  const int j = within / heads;
  const int kv0 = j * C::BKV;
  const SeqView sv = seq_view<VARLEN>(lay, bh);
  if (VARLEN && !sv.ok && kv0 == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadSeqlens);
  if (kv0 >= sv.nk) return;  // past the end of a shorter (or rejected) sequence: the whole CTA leaves
  const int Nq = sv.nq, Nk = sv.nk;
  const int off = VARLEN ? Nk - Nq : 0;  // causal (bottom-right): key visible iff key <= query + off
  const int n_q = (Nq + C::BQ - 1) / C::BQ;
  // causal: the first query that sees key kv0 is kv0 - off
  const int i_begin = CAUSAL ? (kv0 - off <= 0 ? 0 : (kv0 - off) / C::BQ) : 0;
  // Block-sparse: query tile i meets this key tile iff its mask byte
  // (128 x 128 blocks, [mask_heads, n_q, n_q]) is non-zero.
  const uint8_t* mcol = SPARSE ? block_mask + (long long)(mask_heads == 1 ? 0 : bh) * n_q * n_q + j : nullptr;
  auto next_tile = [&](int i) {  // the first visited query tile >= i (n_q if none)
    if constexpr (SPARSE) {
      while (i < n_q && mcol[(long long)i * n_q] == 0) ++i;
    }
    return i;
  };
  int* n_visit = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
  if (SPARSE && warp == 0) {  // count the visited query tiles, 32 at a time
    int cnt = 0;
    for (int b = i_begin; b < n_q; b += 32) {
      const int i = b + lane;
      cnt += __popc(__ballot_sync(0xffffffffu, i < n_q && mcol[(long long)i * n_q] != 0));
    }
    if (lane == 0) *n_visit = cnt;
  }

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int b = 0; b < C::QS; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 2);  // dV (reads dO) and dK (reads Q) issuers
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 4 * C::CWG);   // every compute warp
    mbar_init(p_full, 4 * C::CWG);
    mbar_init(pt_empty, 1);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 4 * C::CWG);
    mbar_init(dkdv_done, 2);
    for (int b = 0; b < 2; ++b) mbar_init(&drain[b], 1);
    for (int b = 0; b < C::CWG; ++b) {
      mbar_init(&ld_full[b], 4);   // the 4 warps of a compute warpgroup
      mbar_init(&ld_empty[b], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
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
  const int n_it = SPARSE ? *n_visit : n_q - i_begin;  // query tiles visited

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
      for (int s = 0; s < C::SLABS; ++s) {
        const int2 ck = sv.kcoord(kv0);
        tma_load_3d(sK + s * C::SLAB, &tm_k, kv_full, s * 64, ck.x, ck.y);
        tma_load_3d(sV + s * C::SLAB, &tm_v, kv_full, s * 64, ck.x, ck.y);
      }
      int issued = 0;
      int i_sp = next_tile(i_begin);  // block-sparse: the query tile of iteration it
      for (int it = 0; it < n_it; ++it) {
        const int b = it % C::QS;
        const uint32_t use = (uint32_t)(it / C::QS);
        if (!mbar_wait(&q_empty[b], (use & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
        mbar_arrive_expect_tx(&q_full[b], 2 * C::TILE);
        const int q0 = (SPARSE ? i_sp : i_begin + it) * C::BQ;
        if constexpr (SPARSE) i_sp = next_tile(i_sp + 1);
        for (int s = 0; s < C::SLABS; ++s) {
          const int2 cq = sv.qcoord(q0);
          tma_load_3d(sQ + b * C::TILE + s * C::SLAB, &tm_q, &q_full[b], s * 64, cq.x, cq.y);
          tma_load_3d(sDO + b * C::TILE + s * C::SLAB, &tm_do, &q_full[b], s * 64, cq.x, cq.y);
        }
        issued = it + 1;
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        drain_wait(kv_full, 0);
        for (int it = issued - C::QS < 0 ? 0 : issued - C::QS; it < issued; ++it)
          drain_wait(&q_full[it % C::QS], (uint32_t)((it / C::QS) & 1));
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    //   warp 1: S^T(i) = K Q_i^T as soon as the compute warps hold S^T(i-1)
    //           in registers, and dV += P^T(i) dO_i (P^T from shared memory)
    //   warp 2: dP^T(i) = V dO_i^T and dK += dS^T(i) Q_i, dS^T read from the
    //           dP^T columns it overwrote (so dK(i) precedes dP^T(i+1) on the
    //           same issuing thread)
    if (lane == 0) {
      const bool first_pair = warp == 1;
      constexpr uint32_t kIdT = idesc_f16(128, C::BQ, BF16, false, false);  // K-major A and B
      constexpr uint32_t kIdAcc = idesc_f16(128, D, BF16, false, true);    // K-major A, MN-major B
      const uint32_t aKV = smem_u32(first_pair ? sK : sV);
      const uint32_t aQD = smem_u32(first_pair ? sQ : sDO);   // B of S^T / dP^T
      const uint32_t aB2 = smem_u32(first_pair ? sDO : sQ);   // B of dV / dK
      const uint32_t aPT = smem_u32(sPT);
      const uint32_t col_t = first_pair ? C::COL_S : C::COL_DP;
      auto issue_t = [&](int qs) {  // S^T or dP^T of the tile in stage qs
        const uint64_t da = sdesc_sw128(aKV, 16, 1024);
        const uint64_t db = sdesc_sw128(aQD + qs * C::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (kk >> 2) * C::SLAB + (kk & 3) * 32;
          mma_ss(tmem + col_t, sdesc_advance(da, o), sdesc_advance(db, o), kIdT, kk > 0);
        }
      };
      auto issue_dv = [&](int qs, bool first) {  // dV += P^T dO, P^T from shared memory
        const uint64_t da = sdesc_sw128(aPT, 16, 1024);
        const uint64_t db = sdesc_sw128(aB2 + qs * C::TILE, C::SLAB, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::PT_SLAB + (kk & 3) * 32;
          mma_ss(tmem + C::COL_DV, sdesc_advance(da, oa), sdesc_advance(db, kk * 2048), kIdAcc, !(first && kk == 0));
        }
      };
      auto issue_dk = [&](int qs, bool first) {  // dK += dS^T Q, dS^T from TMEM
        const uint64_t db = sdesc_sw128(aB2 + qs * C::TILE, C::SLAB, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk) {
          // query columns 16kk .. 16kk+15: warpgroup kk/2 wrote them as 16-bit
          // pairs from its first column, 8 columns per 16 queries
          const uint32_t a = tmem + C::COL_DP + 32 * (kk >> 1) + 8 * (kk & 1);
          mma_ts(tmem + C::COL_DK, a, sdesc_advance(db, kk * 2048), kIdAcc, !(first && kk == 0));
        }
      };
      bool ok = mbar_wait(kv_full, 0, abort_flag, status, kStatusTimeout);
      if (ok && n_it > 0) {
        ok = mbar_wait(&q_full[0], 0, abort_flag, status, kStatusTimeout);
        if (ok) {
          tc_fence_after();
          issue_t(0);
          mma_commit(first_pair ? s_full : dp_full);
        }
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int qs = it % C::QS;
        const int qn = (it + 1) % C::QS;
        const uint32_t qpar = ((it + 1) / C::QS) & 1;
        if (first_pair) {
          if (it + 1 < n_it) {
            if (!(ok = mbar_wait(s_empty, it & 1, abort_flag, status, kStatusTimeout))) break;
            if (!(ok = mbar_wait(&q_full[qn], qpar, abort_flag, status, kStatusTimeout))) break;
            tc_fence_after();
            issue_t(qn);
            mma_commit(s_full);
          }
          if (!(ok = mbar_wait(p_full, it & 1, abort_flag, status, kStatusTimeout))) break;
          tc_fence_after();
          issue_dv(qs, it == 0);
          mma_commit(pt_empty);
          mma_commit(&q_empty[qs]);
        } else {
          if (!(ok = mbar_wait(ds_full, it & 1, abort_flag, status, kStatusTimeout))) break;
          tc_fence_after();
          issue_dk(qs, it == 0);
          mma_commit(&q_empty[qs]);
          if (it + 1 < n_it) {
            if (!(ok = mbar_wait(&q_full[qn], qpar, abort_flag, status, kStatusTimeout))) break;
            tc_fence_after();
            issue_t(qn);
            mma_commit(dp_full);
          }
        }
      }
      if (ok) {
        mma_commit(dkdv_done);
        if (first_pair) count_score_blocks(status, kCountBackward, (unsigned long long)n_it * 4ull);
      } else {  // every MMA this thread issued must finish before TMEM is freed
        mma_commit(&drain[warp - 1]);
        drain_wait(&drain[warp - 1], 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute: P^T, dS^T
    constexpr int QW = C::BQ / C::CWG;  // query columns per warpgroup
    constexpr int NC = QW / 16;         // 16-column chunks per warpgroup
    const int h = (warp >> 2) - 1;      // query columns [QW h, QW (h + 1))
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int key = kv0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    float* sNL = sLD + h * 2 * QW;  // this warpgroup's columns: -LSE log2e, then -D
    float* sND = sNL + QW;
    // P^T of this warpgroup's queries: slab (QW h) / 64, from column (QW h) % 64
    uint8_t* ptslab = sPT + ((QW * h) / 64) * C::PT_SLAB;
    const int ptcol = (QW * h) % 64;
    // LSE and D of query column QW h + r (r < QW), loaded one tile ahead and
    // left untouched until they are staged, so the loads' latency is hidden.
    float pre_l = -pos_inf(), pre_d = 0.f;  // padding query: P = 0
    auto fetch = [&](int i) {
      const int q = i * C::BQ + QW * h + r;
      pre_l = -pos_inf();
      pre_d = 0.f;
      if (r < QW && q < Nq) {
        pre_l = lse[sv.qflat(q)];
        pre_d = delta[sv.qflat(q)];
      }
    };
    int i_sp = next_tile(i_begin);  // block-sparse: the query tile of iteration it
    if (n_it > 0) fetch(SPARSE ? i_sp : i_begin);
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int i = SPARSE ? i_sp : i_begin + it;
      const int q0 = i * C::BQ;
      // Dropout: keep bits of this thread's key for the warpgroup's QW query
      // columns (bit c <-> column c), drawn while S^T(i) is computed.
      uint32_t kw = 0u;
      if constexpr (DROP) kw = key_keep_words(key, q0 + QW * h, QW, lane, bh, drop).x;
      // the staged values of the previous tile have been read by every warp of the warpgroup
      if (it > 0 && !(ok = warp_wait(&ld_empty[h], (it - 1) & 1, abort_flag, status))) break;
      if (r < QW) {
        sNL[r] = pre_l == -pos_inf() ? -pos_inf() : -pre_l * kLog2e;  // a row with no visible key: P = 0
        sND[r] = -pre_d;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ld_full[h]);
      if (!(ok = warp_wait(&ld_full[h], it & 1, abort_flag, status))) break;
      int i_next = i + 1;
      if constexpr (SPARSE) i_next = next_tile(i + 1);
      if (it + 1 < n_it) fetch(i_next);
      // ---- pass 1: S^T into registers (S^T(i+1) may then be issued), P^T into shared memory
      if (!(ok = warp_wait(s_full, it & 1, abort_flag, status))) break;
      tc_fence_after();
      float p[NC][16];
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) tmem_ld16(lane_base + C::COL_S + QW * h + 16 * sc, p[sc]);
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) tmem_ld_wait(p[sc]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
      uint32_t pk[NC][8];
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) {
        const int col = 16 * sc;  // first query column of this chunk within the warpgroup's columns
        const int c0 = q0 + QW * h + col;
        const bool need_mask = (CAUSAL && c0 + off < kv0 + C::BKV - 1) || (kv0 + C::BKV > Nk);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 2 * e;
          const float2 nl = *reinterpret_cast<const float2*>(sNL + col + c);
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(p[sc][c], p[sc][c + 1]), sc2, f2_pack(nl.x, nl.y)), x0, x1);
          float p0, p1;
          if (e < C::POLY_PAIRS) {
            exp2_poly2(x0, x1, p0, p1);
            if (nl.x == -pos_inf()) p0 = 0.f;  // padding query (2^-125, not 0, from the polynomial)
            if (nl.y == -pos_inf()) p1 = 0.f;
          } else {
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
          }
          if (need_mask) {
            if (key >= Nk || (CAUSAL && key > c0 + c + off)) p0 = 0.f;
            if (key >= Nk || (CAUSAL && key > c0 + c + 1 + off)) p1 = 0.f;
          }
          p[sc][c] = p0;
          p[sc][c + 1] = p1;
          pk[sc][e] = pack2(p0, p1, BF16);
          if constexpr (DROP) {  // dV takes the kept entries (scaled by the keep scale when stored)
            const uint32_t b = kw >> (col + c);
            pk[sc][e] &= ((b & 1u) ? 0x0000ffffu : 0u) | ((b & 2u) ? 0xffff0000u : 0u);
          }
        }
      }
      // the P^T buffer is free once dV(i-1) has read it
      if (it > 0 && !(ok = warp_wait(pt_empty, (it - 1) & 1, abort_flag, status))) break;
#pragma unroll
      for (int sc = 0; sc < NC; ++sc)
#pragma unroll
        for (int u = 0; u < 2; ++u)
          *reinterpret_cast<uint4*>(ptslab + sw128_offset(r, ptcol + 16 * sc + 8 * u)) =
              make_uint4(pk[sc][4 * u], pk[sc][4 * u + 1], pk[sc][4 * u + 2], pk[sc][4 * u + 3]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      // ---- pass 2: dS^T = P^T * (dP^T - D), written over dP^T
      if (!(ok = warp_wait(dp_full, it & 1, abort_flag, status))) break;
      tc_fence_after();
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) {
        const int col = 16 * sc;
        float dp[16];
        tmem_ld16(lane_base + C::COL_DP + QW * h + col, dp);
        tmem_ld_wait(dp);
        uint32_t dk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 2 * e;
          const float2 nd = *reinterpret_cast<const float2*>(sND + col + c);
          // dropout: dS = P (Z c dP - D), Z the keep bit and c the keep scale
          uint64_t t2;
          if constexpr (DROP) {
            const uint32_t b = kw >> (col + c);
            t2 = f2_fma(f2_pack(dp[c], dp[c + 1]),
                        f2_pack((b & 1u) ? drop.keep_scale : 0.f, (b & 2u) ? drop.keep_scale : 0.f),
                        f2_pack(nd.x, nd.y));
          } else {
            t2 = f2_add(f2_pack(dp[c], dp[c + 1]), f2_pack(nd.x, nd.y));
          }
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p[sc][c], p[sc][c + 1]), t2), d0, d1);
          dk[e] = pack2(d0, d1, BF16);
        }
        // columns [QW h + col/2, +8) of this warpgroup's own columns were read in chunk sc/2 <= sc
        tmem_st8(lane_base + C::COL_DP + QW * h + 8 * sc, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(ds_full);
        mbar_arrive(&ld_empty[h]);
      }
      if constexpr (SPARSE) i_sp = i_next;
    }
    // ------------------------------------------------------------ epilogue
    // Warpgroups 0 and 1 stage the two 64-feature halves of dV in the Q
    // stages, warpgroups 2 and 3 those of dK * scale in the dO stages; each
    // stores its slab with TMA (rows past N and features past dh fall outside
    // the tensor maps).  Every warp reaches its warpgroup's barrier once.
    const bool is_dk = h >= 2;
    const int half = h & 1;
    const bool has_half = 64 * half < D;
    if (ok && n_it > 0) ok = warp_wait(dkdv_done, 0, abort_flag, status);
    if (ok) tc_fence_after();
    if constexpr (VARLEN) {
      // Packed batches: per-row stores (a tile's last rows can belong to the
      // next sequence); a key tile no query sees writes zeros.
      if (ok && has_half && 64 * half < dh) {
        uint4* dst = reinterpret_cast<uint4*>(is_dk ? dk : dv) + sv.kflat(key) * (dh / 8) + 8 * half;
        const int cols = min(64, dh - 64 * half);
        if (n_it > 0) {
          store_rows_from_tmem<64, BF16>(lane_base + (is_dk ? C::COL_DK : C::COL_DV) + 64 * half, dst, key < Nk,
                                         is_dk ? scale : (DROP ? drop.keep_scale : 1.f), cols);
        } else if (key < Nk) {
          for (int q = 0; q < cols / 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    } else {
      uint8_t* stage = (is_dk ? sDO : sQ) + half * C::SLAB;
      if (ok && has_half)
        stage_rows_from_tmem<64, BF16>(lane_base + (is_dk ? C::COL_DK : C::COL_DV) + 64 * half, stage, r,
                                       is_dk ? scale : (DROP ? drop.keep_scale : 1.f), n_it == 0);
      fence_async_smem();
      named_barrier_sync(1 + h, 128);
      if (r == 0 && ok && has_half && !*abort_flag && 64 * half < dh) {
        tma_store_3d(is_dk ? &tm_dk : &tm_dv, stage, 64 * half, kv0, bh);
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

// ---------------------------------------------------------------- dQ
template <int D>
struct DqCfg : SplitCfg<D> {
  using B = SplitCfg<D>;
  static constexpr int POLY_PAIRS = 0;  // as DkdvSplitCfg
  static constexpr int CWG = 4;         // compute warpgroups, 32 key columns each
  static constexpr int THREADS = 128 + 128 * CWG;
  // K_j is read by S(j) and, a tile later, by dQ(j); V_j only by dP(j): K
  // and V have rings of their own so that a K slot held until dQ(j) never
  // delays the next tiles' loads.
  static constexpr int NK = 3;                     // K ring slots
  static constexpr int NV = 2;                     // V ring slots (slot 1 first stages Q)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = NK * B::TILE;
  static constexpr int OFF_DO = OFF_V + NV * B::TILE;  // dO, the A operand of dP for the whole CTA
  static constexpr int OFF_BAR = OFF_DO + B::TILE;
  // q_full, qa_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full, s_empty, dp_full, dp_empty,
  // ds_full, ds_empty, dq_full, drain[3]
  static constexpr int NBAR = 2 + 2 * NK + 2 * NV + 10;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr uint32_t COL_QA = 0;            // Q as 16-bit pairs (A operand), D/2 columns
  static constexpr uint32_t COL_S = 64;            // 128
  static constexpr uint32_t COL_DP = 192;          // 128
  static constexpr uint32_t COL_DQ = 320;          // D
  static constexpr uint32_t COL_DS = 320 + D;      // dS as 16-bit pairs (A operand of dQ), 64 columns
  static_assert(COL_DS + 64 <= B::TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL, bool BF16, bool SPARSE, bool VARLEN, bool DROP>
__global__ void __launch_bounds__(DqCfg<D>::THREADS, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     void* __restrict__ dq, const float* __restrict__ lse, const float* __restrict__ delta,
                     SeqLayout lay, int BH, int n_qblocks, int dh, float scale, float scale_log2,
                     const uint8_t* __restrict__ block_mask, int mask_heads, DropParams drop, int group,
                     unsigned int* status) {
  using C = DqCfg<D>;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = sV + C::TILE;  // Q staging in V slot 1 until V_1 is loaded
  uint8_t* sDO = smem + C::OFF_DO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* qa_full = q_full + 1;
  uint64_t* k_full = qa_full + 1;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* s_full = v_empty + C::NV;
  uint64_t* s_empty = s_full + 1;    // every compute warp holds S(j) in registers
  uint64_t* dp_full = s_empty + 1;
  uint64_t* dp_empty = dp_full + 1;  // every compute warp holds dP(j) (as dS) in registers
  uint64_t* ds_full = dp_empty + 1;  // dS(j) written to its TMEM columns
  uint64_t* ds_empty = ds_full + 1;  // dQ(j) has read dS(j)
  uint64_t* dq_full = ds_empty + 1;
  uint64_t* drain = dq_full + 1;     // [3]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heads in groups whose K and V fit in about half of L2; inside a group the
  // heaviest query tiles (the last ones, under the causal mask) first.
  const int gi = blockIdx.x / (group * n_qblocks);
  const int heads = min(group, BH - gi * group);
  const int within = blockIdx.x - gi * group * n_qblocks;
  const int bh = gi * group + within % heads;
  const int qb = n_qblocks - 1 - within / heads;
  const int q0 = qb * C::BQ;
  const SeqView sv = seq_view<VARLEN>(lay, bh);
  if (VARLEN && !sv.ok && q0 == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadSeqlens);
  if (q0 >= sv.nq) return;  // past the end of a shorter (or rejected) sequence: the whole CTA leaves
  const int Nq = sv.nq, Nk = sv.nk;
  const int off = VARLEN ? Nk - Nq : 0;  // causal (bottom-right): key visible iff key <= query + off
  const int n_kv = (Nk + C::BKV - 1) / C::BKV;
  const int n_k = CAUSAL ? causal_key_tiles(q0 + C::BQ - 1, off, n_kv, C::BKV) : n_kv;  // key tiles in range
  // Block-sparse: key tile j is visited iff this query tile's mask byte for it is non-zero.
  const uint8_t* mrow =
      SPARSE ? block_mask + (long long)(mask_heads == 1 ? 0 : bh) * n_kv * n_kv + (long long)qb * n_kv : nullptr;
  auto next_tile = [&](int j) {  // the first visited key tile >= j (n_k if none)
    if constexpr (SPARSE) {
      while (j < n_k && mrow[j] == 0) ++j;
    }
    return j;
  };
  int* n_visit = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
  if (SPARSE && warp == 0) {  // count the visited key tiles, 32 at a time
    int cnt = 0;
    for (int b = 0; b < n_k; b += 32) cnt += __popc(__ballot_sync(0xffffffffu, b + lane < n_k && mrow[b + lane] != 0));
    if (lane == 0) *n_visit = cnt;
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(qa_full, 4);  // the 4 warps of compute warpgroup 0
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 4 * C::CWG);  // every compute warp
    mbar_init(dp_full, 1);
    mbar_init(dp_empty, 4 * C::CWG);
    mbar_init(ds_full, 4 * C::CWG);
    mbar_init(ds_empty, 1);
    mbar_init(dq_full, 1);
    for (int b = 0; b < 3; ++b) mbar_init(&drain[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
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
  const int n = SPARSE ? *n_visit : n_k;  // key tiles visited

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::TILE);
      for (int s = 0; s < C::SLABS; ++s) {
        const int2 cq = sv.qcoord(q0);
        tma_load_3d(sQ + s * C::SLAB, &tm_q, q_full, s * 64, cq.x, cq.y);
        tma_load_3d(sDO + s * C::SLAB, &tm_do, q_full, s * 64, cq.x, cq.y);
      }
      int k_issued = 0, v_issued = 0;
      for (int jt = 0, j = next_tile(0); jt < n; ++jt, j = next_tile(j + 1)) {  // K, V of each visited tile
        const int ks = jt % C::NK, vs = jt % C::NV;
        if (!mbar_wait(&k_empty[ks], ((jt / C::NK) & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
        mbar_arrive_expect_tx(&k_full[ks], C::TILE);
        const int2 ck = sv.kcoord((SPARSE ? j : jt) * C::BKV);
        for (int s = 0; s < C::SLABS; ++s)
          tma_load_3d(sK + ks * C::TILE + s * C::SLAB, &tm_k, &k_full[ks], s * 64, ck.x, ck.y);
        k_issued = jt + 1;
        // V slot 1 holds the staged Q until warpgroup 0 has copied it into TMEM
        if (jt == 1 && !mbar_wait(qa_full, 0, abort_flag, status, kStatusTimeout)) break;
        if (!mbar_wait(&v_empty[vs], ((jt / C::NV) & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
        mbar_arrive_expect_tx(&v_full[vs], C::TILE);
        for (int s = 0; s < C::SLABS; ++s)
          tma_load_3d(sV + vs * C::TILE + s * C::SLAB, &tm_v, &v_full[vs], s * 64, ck.x, ck.y);
        v_issued = jt + 1;
      }
      if (*abort_flag) {
        drain_wait(q_full, 0);
        for (int jt = k_issued - C::NK < 0 ? 0 : k_issued - C::NK; jt < k_issued; ++jt)
          drain_wait(&k_full[jt % C::NK], (uint32_t)((jt / C::NK) & 1));
        for (int jt = v_issued - C::NV < 0 ? 0 : v_issued - C::NV; jt < v_issued; ++jt)
          drain_wait(&v_full[jt % C::NV], (uint32_t)((jt / C::NV) & 1));
      }
    }
  } else if (warp >= 1 && warp <= 3) {
    // ------------------------------------------------------------ MMA issuers
    // One thread issues about one MMA per ~100 cycles, so each product has
    // a thread of its own:
    //   warp 1: S(j) = Q K_j^T (Q from TMEM) once S(j-1) is in registers
    //   warp 2: dP(j) = dO V_j^T (dO from shared memory) once dP(j-1) is
    //   warp 3: dQ += dS(j) K_j once dS(j) is written (dS from TMEM)
    if (lane == 0) {
      constexpr uint32_t kIdT = idesc_f16(128, C::BKV, BF16, false, false);  // K-major A and B
      constexpr uint32_t kIdDq = idesc_f16(128, D, BF16, false, true);       // A from TMEM, MN-major B
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      const uint32_t aDO = smem_u32(sDO);
      bool ok = true;
      if (warp == 1) {
        ok = mbar_wait(qa_full, 0, abort_flag, status, kStatusTimeout);
        for (int jt = 0; ok && jt < n; ++jt) {
          if (jt > 0 && !(ok = mbar_wait(s_empty, (jt - 1) & 1, abort_flag, status, kStatusTimeout))) break;
          if (!(ok = mbar_wait(&k_full[jt % C::NK], (jt / C::NK) & 1, abort_flag, status, kStatusTimeout))) break;
          tc_fence_after();
          const uint64_t db = sdesc_sw128(aK + (jt % C::NK) * C::TILE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * C::SLAB + (kk & 3) * 32;
            mma_ts(tmem + C::COL_S, tmem + C::COL_QA + 8 * kk, sdesc_advance(db, o), kIdT, kk > 0);
          }
          mma_commit(s_full);
        }
      } else if (warp == 2) {
        ok = mbar_wait(q_full, 0, abort_flag, status, kStatusTimeout);
        for (int jt = 0; ok && jt < n; ++jt) {
          if (jt > 0 && !(ok = mbar_wait(dp_empty, (jt - 1) & 1, abort_flag, status, kStatusTimeout))) break;
          if (!(ok = mbar_wait(&v_full[jt % C::NV], (jt / C::NV) & 1, abort_flag, status, kStatusTimeout))) break;
          tc_fence_after();
          const uint64_t da = sdesc_sw128(aDO, 16, 1024);
          const uint64_t db = sdesc_sw128(aV + (jt % C::NV) * C::TILE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * C::SLAB + (kk & 3) * 32;
            mma_ss(tmem + C::COL_DP, sdesc_advance(da, o), sdesc_advance(db, o), kIdT, kk > 0);
          }
          mma_commit(dp_full);
          mma_commit(&v_empty[jt % C::NV]);
        }
      } else {
        for (int jt = 0; ok && jt < n; ++jt) {
          if (!(ok = mbar_wait(ds_full, jt & 1, abort_flag, status, kStatusTimeout))) break;
          tc_fence_after();
          const uint64_t db = sdesc_sw128(aK + (jt % C::NK) * C::TILE, C::SLAB, 1024);
#pragma unroll
          for (int kk = 0; kk < C::BKV / 16; ++kk)
            mma_ts(tmem + C::COL_DQ, tmem + C::COL_DS + 8 * kk, sdesc_advance(db, kk * 2048), kIdDq,
                   !(jt == 0 && kk == 0));
          mma_commit(ds_empty);
          mma_commit(&k_empty[jt % C::NK]);  // K_j: S(j) finished before dS(j) existed
        }
        if (ok) mma_commit(dq_full);
      }
      if (!ok) {  // every MMA this thread issued must finish before TMEM is freed
        mma_commit(&drain[warp - 1]);
        drain_wait(&drain[warp - 1], 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute: P, dS
    constexpr int KW = C::BKV / C::CWG;  // key columns per warpgroup
    constexpr int NC = KW / 16;          // 16-column chunks per warpgroup
    const int h = (warp >> 2) - 1;       // key columns [KW h, KW (h + 1)) of every tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int q = q0 + r;            // this thread's query row (TMEM lane)
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = true;
    if (h == 0) {  // Q of this row into TMEM as 16-bit pairs (the A operand of S)
      if ((ok = warp_wait(q_full, 0, abort_flag, status))) {
#pragma unroll
        for (int s = 0; s < C::SLABS; ++s) {
          uint32_t v[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(sQ + s * C::SLAB + sw128_offset(r, 8 * u));
            v[4 * u] = x.x;
            v[4 * u + 1] = x.y;
            v[4 * u + 2] = x.z;
            v[4 * u + 3] = x.w;
          }
          tmem_st32(lane_base + C::COL_QA + 32 * s, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(qa_full);
      }
    }
    const long long frow = sv.qflat(q);
    float nl = -pos_inf(), nd = 0.f;  // padding rows: P = 0
    if (q < Nq) {
      const float lq = lse[frow];
      nl = lq == -pos_inf() ? -pos_inf() : -lq * kLog2e;
      nd = -delta[frow];
    }
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    const uint64_t nl2 = f2_pack(nl, nl);
    const uint64_t nd2 = f2_pack(nd, nd);
    for (int jt = 0, j = next_tile(0); ok && jt < n; ++jt, j = next_tile(j + 1)) {
      const int kb = (SPARSE ? j : jt) * C::BKV + KW * h;  // first key of this warpgroup's columns
      // Dropout: keep bits of this row for the warpgroup's KW key columns
      // (pair i: bits i and 16 + i), drawn while S(j) is computed.
      uint32_t kw[1] = {0u};
      if constexpr (DROP) tile_keep_bits<1>(kw, kb, q, bh, drop.offset, drop.k0, drop.k1, drop.t);
      if (!(ok = warp_wait(s_full, jt & 1, abort_flag, status))) break;
      tc_fence_after();
      float p[NC][16];
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) tmem_ld16(lane_base + C::COL_S + KW * h + 16 * sc, p[sc]);
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) tmem_ld_wait(p[sc]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) {
        const int k0 = kb + 16 * sc;
        const bool need_mask = (CAUSAL && k0 + 15 > q0 + off) || (k0 + 16 > Nk);
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(p[sc][c], p[sc][c + 1]), sc2, nl2), x0, x1);
          float p0, p1;
          if ((c >> 1) < C::POLY_PAIRS) {
            exp2_poly2(x0, x1, p0, p1);
            if (q >= Nq) p0 = p1 = 0.f;  // padding rows (the polynomial gives 2^-125, not 0, at -inf)
          } else {
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
          }
          if (need_mask) {
            if (k0 + c >= Nk || (CAUSAL && k0 + c > q + off)) p0 = 0.f;
            if (k0 + c + 1 >= Nk || (CAUSAL && k0 + c + 1 > q + off)) p1 = 0.f;
          }
          p[sc][c] = p0;
          p[sc][c + 1] = p1;
        }
      }
      if (!(ok = warp_wait(dp_full, jt & 1, abort_flag, status))) break;
      tc_fence_after();
      uint32_t pk[NC][8];
      // both chunks' loads in flight before one wait (the same change in the dK/dV
      // kernel's dS pass measured 2-5% slower there)
      float dpa[NC][16];
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) tmem_ld16(lane_base + C::COL_DP + KW * h + 16 * sc, dpa[sc]);
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) tmem_ld_wait(dpa[sc]);
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) {
        const float* dp = dpa[sc];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float d0, d1;
          uint64_t t2;  // dP - D, or with dropout Z c dP - D (Z the keep bit, c the keep scale)
          if constexpr (DROP) {
            const int pi = 8 * sc + e;  // pair of keys kb + 2 pi, kb + 2 pi + 1
            t2 = f2_fma(f2_pack(dp[2 * e], dp[2 * e + 1]),
                        f2_pack(((kw[0] >> pi) & 1u) ? drop.keep_scale : 0.f,
                                ((kw[0] >> (16 + pi)) & 1u) ? drop.keep_scale : 0.f),
                        nd2);
          } else {
            t2 = f2_add(f2_pack(dp[2 * e], dp[2 * e + 1]), nd2);
          }
          f2_unpack(f2_mul(f2_pack(p[sc][2 * e], p[sc][2 * e + 1]), t2), d0, d1);
          pk[sc][e] = pack2(d0, d1, BF16);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dp_empty);
      // the dS columns are free once dQ(j-1) has read them
      if (jt > 0 && !(ok = warp_wait(ds_empty, (jt - 1) & 1, abort_flag, status))) break;
      tc_fence_after();
      // keys [KW h + 16 sc, +16) -> 16-bit pairs in columns COL_DS + KW h / 2 + 8 sc
#pragma unroll
      for (int sc = 0; sc < NC; ++sc) tmem_st8(lane_base + C::COL_DS + (KW / 2) * h + 8 * sc, pk[sc]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    // ------------------------------------------------------------ epilogue
    // dQ = scale * (dS K summed over key tiles): warpgroup h writes features
    // [FW h, FW (h + 1)) of its row, those below dh.
    constexpr int FW = D / C::CWG;
    if (ok) ok = warp_wait(dq_full, 0, abort_flag, status);
    if constexpr (SPARSE || VARLEN) {  // a square dense tile always visits at least one key tile
      // no visited key tile (an empty mask row, or rows before the first key
      // under a bottom-right causal mask): dQ = 0
      if (ok && n == 0 && FW * h < dh && q < Nq) {
        uint4* drow = reinterpret_cast<uint4*>(dq) + frow * (dh / 8) + FW * h / 8;
#pragma unroll
        for (int u = 0; u < FW / 8; ++u) drow[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (ok && n > 0 && FW * h < dh) {
      tc_fence_after();
      uint4* drow = reinterpret_cast<uint4*>(dq) + frow * (dh / 8) + FW * h / 8;
      float v[FW];
      if constexpr (FW == 32) {
        tmem_ld32(lane_base + C::COL_DQ + FW * h, v);
      } else {
        tmem_ld16(lane_base + C::COL_DQ + FW * h, v);
      }
      tmem_ld_wait(v);
      uint32_t pk[FW / 2];
#pragma unroll
      for (int e = 0; e < FW / 2; ++e) pk[e] = pack2(v[2 * e] * scale, v[2 * e + 1] * scale, BF16);
      if (q < Nq) {
#pragma unroll
        for (int u = 0; u < FW / 8; ++u) drow[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
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

template <int D, bool CAUSAL, bool BF16, bool SPARSE, bool VARLEN, bool DROP>
cudaError_t launch_dkdv_split_t(const SplitArgs& a, cudaStream_t stream) {
  using C = DkdvSplitCfg<D>;
  auto kern = fa_bwd_dkdv_split_kernel<D, CAUSAL, BF16, SPARSE, VARLEN, DROP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_kt = (a.lay.Nk + C::BKV - 1) / C::BKV;  // packed batches: of the longest sequence
  const long long grid = (long long)n_kt * a.BH;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // Q and dO of a head take 4 * N * D bytes; a group keeps them within ~64 MB of L2.
  const long long per_head = 4LL * a.lay.Nq * D;
  const int group = (int)std::max(1LL, std::min(16LL, (64LL << 20) / (per_head > 0 ? per_head : 1)));
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_do, a.tm_k, a.tm_v, a.tm_dk, a.tm_dv, a.dk,
                                                         a.dv, a.lse, a.delta, a.lay, a.BH, a.dh, a.scale,
                                                         a.scale_log2, a.block_mask, a.mask_heads, a.drop, group,
                                                         a.status);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool BF16, bool SPARSE, bool VARLEN, bool DROP>
cudaError_t launch_dq_t(const SplitArgs& a, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = fa_bwd_dq_kernel<D, CAUSAL, BF16, SPARSE, VARLEN, DROP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qblocks = (a.lay.Nq + C::BQ - 1) / C::BQ;  // packed batches: of the longest sequence
  const long long grid = (long long)n_qblocks * a.BH;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // K and V of a head take 4 * N * D bytes; a group keeps them within ~64 MB of L2.
  const long long per_head = 4LL * a.lay.Nk * D;
  const int group = (int)std::max(1LL, std::min(64LL, (64LL << 20) / (per_head > 0 ? per_head : 1)));
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_do, a.tm_k, a.tm_v, a.dq, a.lse, a.delta, a.lay,
                                                         a.BH, n_qblocks, a.dh, a.scale, a.scale_log2, a.block_mask,
                                                         a.mask_heads, a.drop, group, a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_dkdv_split(int d, bool causal, bool bf16, const SplitArgs& a, cudaStream_t stream) {
#define FA_SPLIT_CASE(DD, CC, BB)                                                               \
  if (d == DD && causal == CC && bf16 == BB)                                                   \
    return a.lay.cu_q   ? launch_dkdv_split_t<DD, CC, BB, false, true, false>(a, stream)        \
           : a.block_mask ? launch_dkdv_split_t<DD, CC, BB, true, false, false>(a, stream)      \
           : a.dropout    ? launch_dkdv_split_t<DD, CC, BB, false, false, true>(a, stream)      \
                          : launch_dkdv_split_t<DD, CC, BB, false, false, false>(a, stream);
  FA_SPLIT_CASE(64, false, false)
  FA_SPLIT_CASE(64, false, true)
  FA_SPLIT_CASE(64, true, false)
  FA_SPLIT_CASE(64, true, true)
  FA_SPLIT_CASE(128, false, false)
  FA_SPLIT_CASE(128, false, true)
  FA_SPLIT_CASE(128, true, false)
  FA_SPLIT_CASE(128, true, true)
#undef FA_SPLIT_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_backward_dq(int d, bool causal, bool bf16, const SplitArgs& a, cudaStream_t stream) {
#define FA_DQ_CASE(DD, CC, BB)                                                                   \
  if (d == DD && causal == CC && bf16 == BB)                                                   \
    return a.lay.cu_q   ? launch_dq_t<DD, CC, BB, false, true, false>(a, stream)                \
           : a.block_mask ? launch_dq_t<DD, CC, BB, true, false, false>(a, stream)              \
           : a.dropout    ? launch_dq_t<DD, CC, BB, false, false, true>(a, stream)              \
                          : launch_dq_t<DD, CC, BB, false, false, false>(a, stream);
  FA_DQ_CASE(64, false, false)
  FA_DQ_CASE(64, false, true)
  FA_DQ_CASE(64, true, false)
  FA_DQ_CASE(64, true, true)
  FA_DQ_CASE(128, false, false)
  FA_DQ_CASE(128, false, true)
  FA_DQ_CASE(128, true, false)
  FA_DQ_CASE(128, true, true)
#undef FA_DQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa

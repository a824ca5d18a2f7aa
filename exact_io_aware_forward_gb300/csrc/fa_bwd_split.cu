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
//   S^T = K Q_i^T, dP^T = V dO_i^T;  P^T and dS^T are written as 16-bit pairs
//   over the first half of each compute warpgroup's own S^T / dP^T columns,
//   where dV += P^T dO_i and dK += dS^T Q_i read them as A operands.
// Warps (384 threads):
//   0      TMA: K, V once; Q_i, dO_i through a ring (2 stages at D = 128).
//   1      TMEM allocation; lane 0 issues S^T(i+1) and dV(i).
//   2      lane 0 issues dP^T(i+1) and dK(i).
//   4-7 / 8-11  compute warpgroup h = 0 / 1: one key row per thread (TMEM
//          lane), query columns [64h, 64h + 64): P^T from S^T and LSE (pass
//          1, P kept in registers), then dS^T from dP^T and D (pass 2).
//   Each issuer orders its own product pair: dV(i) reads P^T(i) from the S^T
//   columns before S^T(i+1) overwrites them (same issuing thread, in order),
//   and likewise dK(i) before dP^T(i+1).  P^T(i) is formed while dK(i-1) and
//   dP^T(i) run, dS^T(i) while dV(i) and S^T(i+1) run.
//
// fa_bwd_dq_kernel -- one CTA per 128-query tile, looping over 128-key tiles.
// Q and dO of the tile are copied once into TMEM as A operands.  TMEM (D = 128):
//   Q 64 | dO 64 | S 128 | dP 128 | dQ 128
//   S = Q K_j^T, dP = dO V_j^T;  dS (16-bit) over the first half of each
//   compute warpgroup's dP columns;  dQ += dS K_j accumulates in TMEM for the
//   whole key loop and is scaled and stored once.
// Warps (384 threads): 0 TMA (Q, dO once; K_j, V_j through a 4-slot ring in
//   the order K0 V0 K1 V1 ...), 1 TMEM allocation and the MMA issuer (order
//   S(0) dP(0) | S(j+1) dQ(j) dP(j+1) | ...), 4-7 / 8-11 compute warpgroups,
//   one query row per thread and key columns [64h, 64h + 64).
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
  static constexpr int QS = D == 128 ? 2 : 4;      // Q / dO stages
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = B::TILE;
  static constexpr int OFF_Q = 2 * B::TILE;        // [QS]
  static constexpr int OFF_DO = OFF_Q + QS * B::TILE;
  static constexpr int OFF_LD = OFF_DO + QS * B::TILE;  // [2 buffers][2: -LSE log2e, -D][128] floats
  static constexpr int OFF_BAR = OFF_LD + 2 * 2 * 128 * 4;
  // kv_full, q_full[QS], q_empty[QS], s_full, dp_full, p_full, ds_full, dkdv_done, drain[2], ld_full[2]
  static constexpr int NBAR = 1 + 2 * QS + 5 + 2 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = 128;
  static constexpr uint32_t COL_DV = 256;
  static constexpr uint32_t COL_DK = 256 + D;
  static_assert(COL_DK + D <= B::TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dkdv_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                             const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                             const float* __restrict__ lse, const float* __restrict__ delta, int N, int BH, int dh,
                             float scale, float scale_log2, int group, unsigned int* status) {
  using C = DkdvSplitCfg<D>;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  float* sLD = reinterpret_cast<float*>(smem + C::OFF_LD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = kv_full + 1;
  uint64_t* q_empty = q_full + C::QS;
  uint64_t* s_full = q_empty + C::QS;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_full = dp_full + 1;
  uint64_t* ds_full = p_full + 1;
  uint64_t* dkdv_done = ds_full + 1;
  uint64_t* drain = dkdv_done + 1;
  uint64_t* ld_full = drain + 2;  // [2]: -LSE log2e and -D of a tile staged by the compute warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heads in groups of `group` (a group's Q and dO fit in about half of L2);
  // inside a group key tile 0 of every head (which meets every query tile
  // under the causal mask) first, then key tile 1, ...
  const int n_kt = (N + C::BKV - 1) / C::BKV;
  const int gi = blockIdx.x / (group * n_kt);
  const int heads = min(group, BH - gi * group);
  const int within = blockIdx.x - gi * group * n_kt;
  const int bh = gi * group + within % heads;
  const int j = within / heads;
  const int kv0 = j * C::BKV;
  const int n_q = (N + C::BQ - 1) / C::BQ;
  const int i_begin = CAUSAL ? kv0 / C::BQ : 0;  // first query tile with a query >= kv0
  const int n_it = n_q - i_begin;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int b = 0; b < C::QS; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 2);  // dV (reads dO) and dK (reads Q) issuers
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 8);   // the 8 compute warps
    mbar_init(ds_full, 8);
    mbar_init(dkdv_done, 2);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(&ld_full[0], 8);
    mbar_init(&ld_full[1], 8);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
      for (int s = 0; s < C::SLABS; ++s) {
        tma_load_3d(sK + s * C::SLAB, &tm_k, kv_full, s * 64, kv0, bh);
        tma_load_3d(sV + s * C::SLAB, &tm_v, kv_full, s * 64, kv0, bh);
      }
      int issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int b = it % C::QS;
        const uint32_t use = (uint32_t)(it / C::QS);
        if (!mbar_wait(&q_empty[b], (use & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
        mbar_arrive_expect_tx(&q_full[b], 2 * C::TILE);
        const int q0 = (i_begin + it) * C::BQ;
        for (int s = 0; s < C::SLABS; ++s) {
          tma_load_3d(sQ + b * C::TILE + s * C::SLAB, &tm_q, &q_full[b], s * 64, q0, bh);
          tma_load_3d(sDO + b * C::TILE + s * C::SLAB, &tm_do, &q_full[b], s * 64, q0, bh);
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
    //   warp 1: S^T(i) = K Q_i^T and dV += P^T(i) dO_i
    //   warp 2: dP^T(i) = V dO_i^T and dK += dS^T(i) Q_i
    if (lane == 0) {
      const bool first_pair = warp == 1;
      constexpr uint32_t kIdT = idesc_f16(128, C::BQ, BF16, false, false);  // K-major A and B
      constexpr uint32_t kIdAcc = idesc_f16(128, D, BF16, false, true);    // A from TMEM, MN-major B
      const uint32_t aKV = smem_u32(first_pair ? sK : sV);
      const uint32_t aQD = smem_u32(first_pair ? sQ : sDO);   // B of S^T / dP^T
      const uint32_t aB2 = smem_u32(first_pair ? sDO : sQ);   // B of dV / dK
      const uint32_t col_t = first_pair ? C::COL_S : C::COL_DP;
      const uint32_t col_acc = first_pair ? C::COL_DV : C::COL_DK;
      uint64_t* t_full = first_pair ? s_full : dp_full;
      uint64_t* a_full = first_pair ? p_full : ds_full;
      auto issue_t = [&](int qs) {  // S^T or dP^T of the tile in stage qs
        const uint64_t da = sdesc_sw128(aKV, 16, 1024);
        const uint64_t db = sdesc_sw128(aQD + qs * C::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * C::SLAB + (kk & 3) * 32) >> 4;
          mma_ss(tmem + col_t, da + o, db + o, kIdT, kk > 0);
        }
      };
      auto issue_acc = [&](int qs, bool first) {  // dV += P^T dO or dK += dS^T Q
        const uint64_t db = sdesc_sw128(aB2 + qs * C::TILE, C::SLAB, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk) {
          // query columns 16kk .. 16kk+15: warpgroup kk/4 wrote them as 16-bit
          // pairs from its first column, 8 columns per 16 queries
          const uint32_t a = tmem + col_t + 64 * (kk >> 2) + 8 * (kk & 3);
          mma_ts(tmem + col_acc, a, db + ((kk * 2048) >> 4), kIdAcc, !(first && kk == 0));
        }
      };
      bool ok = mbar_wait(kv_full, 0, abort_flag, status, kStatusTimeout);
      if (ok && n_it > 0) {
        ok = mbar_wait(&q_full[0], 0, abort_flag, status, kStatusTimeout);
        if (ok) {
          tc_fence_after();
          issue_t(0);
          mma_commit(t_full);
        }
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int qs = it % C::QS;
        if (!(ok = mbar_wait(a_full, it & 1, abort_flag, status, kStatusTimeout))) break;
        tc_fence_after();
        issue_acc(qs, it == 0);
        mma_commit(&q_empty[qs]);
        if (it + 1 < n_it) {
          const int qn = (it + 1) % C::QS;
          if (!(ok = mbar_wait(&q_full[qn], ((it + 1) / C::QS) & 1, abort_flag, status, kStatusTimeout))) break;
          tc_fence_after();
          issue_t(qn);
          mma_commit(t_full);
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
    const int h = (warp >> 2) - 1;  // query columns [64h, 64h + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int key = kv0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    const long long row0 = (long long)bh * N;
    // -LSE*log2(e) and -D of query column 64h + r (r < 64), fetched one tile ahead
    float pre_l = 0.f, pre_d = 0.f;
    auto fetch = [&](int i) {
      const int q = i * C::BQ + 64 * h + r;
      if (r < 64) {
        if (q < N) {
          const float lq = lse[row0 + q];
          pre_l = lq == -pos_inf() ? -pos_inf() : -lq * kLog2e;
          pre_d = -delta[row0 + q];
        } else {  // padding query: P = 0
          pre_l = -pos_inf();
          pre_d = 0.f;
        }
      }
    };
    if (n_it > 0) fetch(i_begin);
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int i = i_begin + it;
      const int q0 = i * C::BQ;
      float* sNL = sLD + (it & 1) * 256;
      float* sND = sNL + 128;
      if (r < 64) {
        sNL[64 * h + r] = pre_l;
        sND[64 * h + r] = pre_d;
      }
      // Buffer it & 1 is rewritten two tiles later, after every compute warp
      // has passed this wait for the next tile, i.e. finished this one.
      __syncwarp();
      if (lane == 0) mbar_arrive(&ld_full[it & 1]);
      if (!(ok = warp_wait(&ld_full[it & 1], (it >> 1) & 1, abort_flag, status))) break;
      if (it + 1 < n_it) fetch(i + 1);
      // ---- pass 1: P^T = exp2(S^T s log2e - LSE log2e), masked
      if (!(ok = warp_wait(s_full, it & 1, abort_flag, status))) break;
      tc_fence_after();
      float p[4][16];
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) {
        const int col = 64 * h + 16 * sc;  // first query column (within the tile) of this chunk
        float s[16];
        tmem_ld16(lane_base + C::COL_S + col, s);
        tmem_ld_wait(s);
        const int c0 = q0 + col;
        const bool need_mask = (CAUSAL && c0 < kv0 + C::BKV - 1) || (kv0 + C::BKV > N);
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 2 * e;
          const float2 nl = *reinterpret_cast<const float2*>(sNL + col + c);
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sc2, f2_pack(nl.x, nl.y)), x0, x1);
          float p0 = ex2_approx(x0);
          float p1 = ex2_approx(x1);
          if (need_mask) {
            if (key >= N || (CAUSAL && key > c0 + c)) p0 = 0.f;
            if (key >= N || (CAUSAL && key > c0 + c + 1)) p1 = 0.f;
          }
          p[sc][c] = p0;
          p[sc][c + 1] = p1;
          pk[e] = pack2(p0, p1, BF16);
        }
        // columns [col/2 ...] of this warpgroup's own half were read in chunk sc/2 <= sc
        tmem_st8(lane_base + C::COL_S + 64 * h + 8 * sc, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      // ---- pass 2: dS^T = P^T * (dP^T - D)
      if (!(ok = warp_wait(dp_full, it & 1, abort_flag, status))) break;
      tc_fence_after();
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) {
        const int col = 64 * h + 16 * sc;
        float dp[16];
        tmem_ld16(lane_base + C::COL_DP + col, dp);
        tmem_ld_wait(dp);
        uint32_t dk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 2 * e;
          const float2 nd = *reinterpret_cast<const float2*>(sND + col + c);
          const uint64_t t2 = f2_add(f2_pack(dp[c], dp[c + 1]), f2_pack(nd.x, nd.y));
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p[sc][c], p[sc][c + 1]), t2), d0, d1);
          dk[e] = pack2(d0, d1, BF16);
        }
        tmem_st8(lane_base + C::COL_DP + 64 * h + 8 * sc, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    // ------------------------------------------------------------ epilogue
    // dV (warpgroup 0, staged in the Q stages) and dK * scale (warpgroup 1,
    // staged in the dO stages), stored with TMA; rows past N and features
    // past dh fall outside the tensor maps.  Every warp reaches the barrier.
    if (ok && n_it > 0) ok = warp_wait(dkdv_done, 0, abort_flag, status);
    if (ok) tc_fence_after();
    uint8_t* stage = h == 0 ? sQ : sDO;
    if (ok) stage_rows_from_tmem<D, BF16>(lane_base + (h == 0 ? C::COL_DV : C::COL_DK), stage, r,
                                          h == 0 ? 1.f : scale, n_it == 0);
    fence_async_smem();
    named_barrier_sync(1 + h, 128);
    if (r == 0 && ok && !*abort_flag)
      store_staged_tile<D>(h == 0 ? &tm_dv : &tm_dk, stage, 0, dh, make_int2(kv0, bh));
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
  static constexpr int NS = D == 128 ? 4 : 8;      // K / V ring slots
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_Q = NS * B::TILE;       // Q and dO staging (copied into TMEM once)
  static constexpr int OFF_DO = OFF_Q + B::TILE;
  static constexpr int OFF_BAR = OFF_DO + B::TILE;
  // q_full, qa_full, ring_full[NS], ring_empty[NS], s_full, s_empty, dp_full, ds_full, dq_full, drain
  static constexpr int NBAR = 2 + 2 * NS + 6;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr uint32_t COL_QA = 0;            // Q as 16-bit pairs (A operand), D/2 columns
  static constexpr uint32_t COL_DOA = D / 2;       // dO likewise
  static constexpr uint32_t COL_S = D;             // 128
  static constexpr uint32_t COL_DP = D + 128;      // 128
  static constexpr uint32_t COL_DQ = D + 256;      // D
  static_assert(COL_DQ + D <= B::TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     void* __restrict__ dq, const float* __restrict__ lse, const float* __restrict__ delta, int N,
                     int BH, int n_qblocks, int dh, float scale, float scale_log2, int group, unsigned int* status) {
  using C = DqCfg<D>;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sRing = smem + C::OFF_RING;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* qa_full = q_full + 1;
  uint64_t* ring_full = qa_full + 1;
  uint64_t* ring_empty = ring_full + C::NS;
  uint64_t* s_full = ring_empty + C::NS;
  uint64_t* s_empty = s_full + 1;
  uint64_t* dp_full = s_empty + 1;
  uint64_t* ds_full = dp_full + 1;
  uint64_t* dq_full = ds_full + 1;
  uint64_t* drain = dq_full + 1;
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
  const int n_kv = (N + C::BKV - 1) / C::BKV;
  const int n = CAUSAL ? causal_key_tiles(q0 + C::BQ - 1, 0, n_kv, C::BKV) : n_kv;  // key tiles visited

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(qa_full, 8);  // the 8 compute warps
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 8);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(dq_full, 1);
    mbar_init(drain, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::TILE);
      for (int s = 0; s < C::SLABS; ++s) {
        tma_load_3d(sQ + s * C::SLAB, &tm_q, q_full, s * 64, q0, bh);
        tma_load_3d(sDO + s * C::SLAB, &tm_do, q_full, s * 64, q0, bh);
      }
      int issued = 0;
      for (int u = 0; u < 2 * n; ++u) {  // K_0, V_0, K_1, V_1, ...
        const int slot = u % C::NS;
        const uint32_t use = (uint32_t)(u / C::NS);
        if (!mbar_wait(&ring_empty[slot], (use & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
        mbar_arrive_expect_tx(&ring_full[slot], C::TILE);
        const CUtensorMap* m = (u & 1) ? &tm_v : &tm_k;
        for (int s = 0; s < C::SLABS; ++s)
          tma_load_3d(sRing + slot * C::TILE + s * C::SLAB, m, &ring_full[slot], s * 64, (u >> 1) * C::BKV, bh);
        issued = u + 1;
      }
      if (*abort_flag) {
        drain_wait(q_full, 0);
        for (int u = issued - C::NS < 0 ? 0 : issued - C::NS; u < issued; ++u)
          drain_wait(&ring_full[u % C::NS], (uint32_t)((u / C::NS) & 1));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdT = idesc_f16(128, C::BKV, BF16, false, false);  // A from TMEM, K-major B
      constexpr uint32_t kIdDq = idesc_f16(128, D, BF16, false, true);       // A from TMEM, MN-major B
      const uint32_t ring = smem_u32(sRing);
      auto slot_of = [](int u) { return u % C::NS; };
      auto par_of = [](int u) { return (uint32_t)((u / C::NS) & 1); };
      // S = Q K_j^T (a = Q) or dP = dO V_j^T (a = dO): tile item u of the ring
      auto issue_t = [&](uint32_t acol, uint32_t dcol, int u) {
        const uint64_t db = sdesc_sw128(ring + slot_of(u) * C::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * C::SLAB + (kk & 3) * 32) >> 4;
          mma_ts(tmem + dcol, tmem + acol + 8 * kk, db + o, kIdT, kk > 0);
        }
      };
      auto issue_dq = [&](int u, bool first) {  // dQ += dS K_j
        const uint64_t db = sdesc_sw128(ring + slot_of(u) * C::TILE, C::SLAB, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BKV / 16; ++kk) {
          const uint32_t a = tmem + C::COL_DP + 64 * (kk >> 2) + 8 * (kk & 3);
          mma_ts(tmem + C::COL_DQ, a, db + ((kk * 2048) >> 4), kIdDq, !(first && kk == 0));
        }
      };
      bool ok = mbar_wait(qa_full, 0, abort_flag, status, kStatusTimeout);
      if (ok && n > 0) {
        ok = mbar_wait(&ring_full[slot_of(0)], par_of(0), abort_flag, status, kStatusTimeout);
        if (ok) {
          tc_fence_after();
          issue_t(C::COL_QA, C::COL_S, 0);
          mma_commit(s_full);
          ok = mbar_wait(&ring_full[slot_of(1)], par_of(1), abort_flag, status, kStatusTimeout);
        }
        if (ok) {
          tc_fence_after();
          issue_t(C::COL_DOA, C::COL_DP, 1);
          mma_commit(dp_full);
          mma_commit(&ring_empty[slot_of(1)]);
        }
      }
      for (int jt = 0; ok && jt < n; ++jt) {
        if (jt + 1 < n) {  // S(j+1) once the compute warps hold S(j) in registers
          if (!(ok = mbar_wait(s_empty, jt & 1, abort_flag, status, kStatusTimeout))) break;
          if (!(ok = mbar_wait(&ring_full[slot_of(2 * jt + 2)], par_of(2 * jt + 2), abort_flag, status,
                               kStatusTimeout)))
            break;
          tc_fence_after();
          issue_t(C::COL_QA, C::COL_S, 2 * jt + 2);
          mma_commit(s_full);
        }
        if (!(ok = mbar_wait(ds_full, jt & 1, abort_flag, status, kStatusTimeout))) break;
        tc_fence_after();
        issue_dq(2 * jt, jt == 0);
        mma_commit(&ring_empty[slot_of(2 * jt)]);
        if (jt + 1 < n) {  // dP(j+1) overwrites dS(j) after dQ(j) has read it (same thread, in order)
          if (!(ok = mbar_wait(&ring_full[slot_of(2 * jt + 3)], par_of(2 * jt + 3), abort_flag, status,
                               kStatusTimeout)))
            break;
          tc_fence_after();
          issue_t(C::COL_DOA, C::COL_DP, 2 * jt + 3);
          mma_commit(dp_full);
          mma_commit(&ring_empty[slot_of(2 * jt + 3)]);
        }
      }
      if (ok) {
        mma_commit(dq_full);
      } else {
        mma_commit(drain);
        drain_wait(drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute: P, dS
    const int h = (warp >> 2) - 1;  // key columns [64h, 64h + 64) of every tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int q = q0 + r;            // this thread's query row (TMEM lane)
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = true;
    // Q (warpgroup 0) or dO (warpgroup 1) of this row into TMEM as 16-bit pairs.
    if (!(ok = warp_wait(q_full, 0, abort_flag, status))) {
    } else {
      const uint8_t* src = h == 0 ? sQ : sDO;
      const uint32_t dcol = h == 0 ? C::COL_QA : C::COL_DOA;
#pragma unroll
      for (int s = 0; s < C::SLABS; ++s) {
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = *reinterpret_cast<const uint4*>(src + s * C::SLAB + sw128_offset(r, 8 * u));
          v[4 * u] = x.x;
          v[4 * u + 1] = x.y;
          v[4 * u + 2] = x.z;
          v[4 * u + 3] = x.w;
        }
        tmem_st32(lane_base + dcol + 32 * s, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(qa_full);
    }
    const long long frow = (long long)bh * N + q;
    float nl = -pos_inf(), nd = 0.f;  // padding rows: P = 0
    if (q < N) {
      const float lq = lse[frow];
      nl = lq == -pos_inf() ? -pos_inf() : -lq * kLog2e;
      nd = -delta[frow];
    }
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    const uint64_t nl2 = f2_pack(nl, nl);
    const uint64_t nd2 = f2_pack(nd, nd);
    for (int jt = 0; ok && jt < n; ++jt) {
      const int kb = jt * C::BKV + 64 * h;  // first key of this warpgroup's columns
      if (!(ok = warp_wait(s_full, jt & 1, abort_flag, status))) break;
      tc_fence_after();
      float p[4][16];
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) tmem_ld16(lane_base + C::COL_S + 64 * h + 16 * sc, p[sc]);
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) tmem_ld_wait(p[sc]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) {
        const int k0 = kb + 16 * sc;
        const bool need_mask = (CAUSAL && k0 + 15 > q0) || (k0 + 16 > N);
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(p[sc][c], p[sc][c + 1]), sc2, nl2), x0, x1);
          float p0 = ex2_approx(x0);
          float p1 = ex2_approx(x1);
          if (need_mask) {
            if (k0 + c >= N || (CAUSAL && k0 + c > q)) p0 = 0.f;
            if (k0 + c + 1 >= N || (CAUSAL && k0 + c + 1 > q)) p1 = 0.f;
          }
          p[sc][c] = p0;
          p[sc][c + 1] = p1;
        }
      }
      if (!(ok = warp_wait(dp_full, jt & 1, abort_flag, status))) break;
      tc_fence_after();
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) {
        float dp[16];
        tmem_ld16(lane_base + C::COL_DP + 64 * h + 16 * sc, dp);
        tmem_ld_wait(dp);
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p[sc][2 * e], p[sc][2 * e + 1]), f2_add(f2_pack(dp[2 * e], dp[2 * e + 1]), nd2)),
                    d0, d1);
          pk[e] = pack2(d0, d1, BF16);
        }
        // the columns written were read in chunk sc/2 <= sc
        tmem_st8(lane_base + C::COL_DP + 64 * h + 8 * sc, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
    }
    // ------------------------------------------------------------ epilogue
    // dQ = scale * (dS K summed over key tiles): warpgroup h writes features
    // [D/2 h, D/2 (h + 1)) of its row, those below dh.
    if (ok) ok = warp_wait(dq_full, 0, abort_flag, status);
    if (ok && n > 0) {
      tc_fence_after();
      uint4* drow = reinterpret_cast<uint4*>(dq) + frow * (dh / 8);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int f0 = (D / 2) * h + 32 * c;  // first feature of this 32-column chunk
        if (f0 >= dh) break;
        float v[32];
        tmem_ld32(lane_base + C::COL_DQ + f0, v);
        tmem_ld_wait(v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack2(v[2 * e] * scale, v[2 * e + 1] * scale, BF16);
        if (q < N) {
#pragma unroll
          for (int u = 0; u < 4; ++u) drow[f0 / 8 + u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
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

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_dkdv_split_t(const SplitArgs& a, cudaStream_t stream) {
  using C = DkdvSplitCfg<D>;
  auto kern = fa_bwd_dkdv_split_kernel<D, CAUSAL, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_kt = (a.N + C::BKV - 1) / C::BKV;
  const long long grid = (long long)n_kt * a.BH;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // Q and dO of a head take 4 * N * D bytes; a group keeps them within ~64 MB of L2.
  const long long per_head = 4LL * a.N * D;
  const int group = (int)std::max(1LL, std::min(16LL, (64LL << 20) / (per_head > 0 ? per_head : 1)));
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_do, a.tm_k, a.tm_v, a.tm_dk, a.tm_dv, a.lse,
                                                         a.delta, a.N, a.BH, a.dh, a.scale, a.scale_log2, group,
                                                         a.status);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_dq_t(const SplitArgs& a, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = fa_bwd_dq_kernel<D, CAUSAL, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qblocks = (a.N + C::BQ - 1) / C::BQ;
  const long long grid = (long long)n_qblocks * a.BH;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // K and V of a head take 4 * N * D bytes; a group keeps them within ~64 MB of L2.
  const long long per_head = 4LL * a.N * D;
  const int group = (int)std::max(1LL, std::min(64LL, (64LL << 20) / (per_head > 0 ? per_head : 1)));
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_do, a.tm_k, a.tm_v, a.dq, a.lse, a.delta, a.N,
                                                         a.BH, n_qblocks, a.dh, a.scale, a.scale_log2, group,
                                                         a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_dkdv_split(int d, bool causal, bool bf16, const SplitArgs& a, cudaStream_t stream) {
#define FA_SPLIT_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_dkdv_split_t<DD, CC, BB>(a, stream);
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
#define FA_DQ_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_dq_t<DD, CC, BB>(a, stream);
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

// dK / dV kernel of the backward pass on sm_103a (stage 2 of fa_backward): the
// kernel template, shared by the translation units that instantiate it
// (fa_bwd.cu: dense and block-sparse; fa_bwd_dropout.cu: dropout;
// fa_bwd_varlen.cu: packed variable-length batches).
//
// Math ("FlashAttention 为什么不需要存下注意力矩阵", jefxiong.cn, section 3.3):
// with G = dO, P = exp(s Q K^T - LSE) recomputed tile by tile on chip,
//   dP = G V^T,  dS = P * (dP - D),  D_i = dO_i . O_i,
//   dV = P^T G,  dK = s dS^T Q,  dQ = s dS K.
// Nothing N x N is stored: P and dS of one (key tile, query tile) pair live
// in TMEM / shared memory only while their products are formed.
//
// One CTA owns one key tile (128 keys, the tcgen05 M dimension) and loops
// over query tiles of BQ rows (64 at d = 128, 128 at d = 64).  Transposed
// products keep the key dimension on TMEM lanes:
//   S^T  = K Q_i^T        [128 x BQ]  TMEM
//   dP^T = V dO_i^T       [128 x BQ]  TMEM
//   P^T  = exp2(S^T s log2e - LSE_i log2e),  dS^T = P^T * (dP^T - D_i)
//                                      -> shared memory, 16-bit, 128B swizzle
//   dV  += P^T dO_i       [128 x d]   TMEM accumulator
//   dK  += dS^T Q_i       [128 x d]   TMEM accumulator
//   dQ_i partial: d = 128: dQ_i^T = K^T dS^T  [128 x 64]  (lane = feature)
//                 d =  64: dQ_i   = dS K      [128 x 64]  (lane = query)
//     double-buffered in TMEM and added into the float32 dq_accum with
//     vector/scalar reductions (red.global.add) by a separate warpgroup.
//
// Warp roles (640 threads):
//   warp 0      TMA: K, V once; Q_i, dO_i through a 3-stage ring (1 at d = 256).
//   warps 1-3   TMEM allocation (warp 1); lane 0 of each issues part of the
//               tcgen05.mma work (one thread can only issue about one MMA per
//               ~100 cycles).  The S^T and dP^T of tile i+1 are issued as soon
//               as the compute warps have pulled tile i's into registers, so
//               the tensor core works on tile i+1 while tile i's P and dS
//               are formed.
//   warps 4-7, 12-15  compute: one key row per thread (TMEM lane), each
//               warpgroup on half of the query columns.  P^T and dS^T have
//               one buffer each (TMEM at d = 128, where dV and dK then read
//               their A operand from TMEM; shared memory at d = 64; dS^T is
//               always in shared memory too, as an operand of the dQ
//               product), written after the math of the next tile once the
//               previous tile's products are done.
//   warps 8-11, 16-19  dQ drain (each warpgroup half of the columns), then
//               half of the epilogue.
// Causal: query tiles entirely above the diagonal are skipped by the loop
// bounds (the whole-block skip of section 4.5); the diagonal tile is
// masked elementwise.  Block-sparse (SPARSE): query tiles whose 128-row
// block does not keep this key tile are skipped as well; a key tile kept by
// no query tile writes dK = dV = 0.
// Dropout (DROP): each entry's keep bit is regenerated from the Philox seed
// and offset (fa_philox.cuh), one generator call per 8 keys of a query: the
// 8 lanes holding those keys each make the call of one query and an 8 x 8 bit
// transpose across the lanes hands every lane the bits of its own key.  The
// dQ drain warps, which share the compute warps' TMEM lanes (keys) and wait
// for most of each tile, draw the bits one tile ahead into shared memory.
// The dV operand is the kept P (scaled by the keep scale in the epilogue)
// and dS^T = P^T * (keep * scale * dP^T - D).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "fa_layout.cuh"
#include "fa_philox.cuh"
#include "fa_ptx.cuh"

namespace fa {

namespace {

__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000u); }

// D = 256: dK and dV of 128 keys x 256 features would fill all 512 TMEM
// columns, so each (key tile, head) is processed by NP = 2 CTAs, one per
// 128-feature half of dK, dV and dQ (DA = 128 accumulator columns).  Both
// recompute S^T and dP^T over all 256 features; K, V and a single Q / dO
// stage fill shared memory.
template <int D>
struct BwdCfg {
  static constexpr int BKV = 128;                   // keys per CTA (MMA M)
  static constexpr int BQ = D == 64 ? 128 : 64;     // query rows per iteration
  static constexpr bool DQT = D != 64;              // dQ computed transposed
  static constexpr int DA = D == 256 ? 128 : D;     // features of dK / dV / dQ per CTA
  static constexpr int NP = D / DA;                 // CTAs per (key tile, head)
  static constexpr int SLABS = D / 64;
  static constexpr int KV_SLAB = BKV * 128;         // 128 rows x 64 cols x 16 bit
  static constexpr int KV_TILE = SLABS * KV_SLAB;
  static constexpr int Q_SLAB = BQ * 128;           // BQ rows x 64 cols x 16 bit
  static constexpr int Q_TILE = SLABS * Q_SLAB;
  static constexpr int PT_SLAB = BKV * 128;         // 128 key rows x 64 query cols
  static constexpr int PT_TILE = (BQ / 64) * PT_SLAB;
  static constexpr int PS = 1;                      // P^T / dS^T buffers
  static constexpr int QS = D == 256 ? 1 : 3;  // Q / dO stages (4 at d = 128 measured 0.6% slower)
  // One stage (D = 256): its slabs outside this CTA's feature half are only
  // read by S^T and dP^T, so they are released and reloaded with the next
  // tile as soon as those products are done (barriers qo_full / qo_empty),
  // while the CTA's own half waits for dK / dV.
  static constexpr bool SPLIT = QS == 1;
  static_assert(!SPLIT || NP == 2, "the split stage pairs two feature halves");
  // d >= 128: P^T and dS^T also go to TMEM (A operands of dV and dK read from
  // TMEM, saving shared-memory bandwidth); dQ then has one TMEM buffer.
  static constexpr bool PT_TMEM = D != 64;
  static constexpr int DQB = PT_TMEM ? 1 : 2;       // dQ TMEM buffers
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;     // [QS] stages
  static constexpr int OFF_DO = OFF_Q + QS * Q_TILE;
  static constexpr int OFF_P = OFF_DO + QS * Q_TILE; // [PS]
  static constexpr int OFF_DS = OFF_P + (PT_TMEM ? 0 : PS * PT_TILE);
  static constexpr int OFF_LD = OFF_DS + PS * PT_TILE;  // [2][2][BQ] floats: LSE*log2e, D
  // dropout keep words [2 buffers][2 compute warpgroups][128 keys] x uint2, drawn by the dQ drain warps
  static constexpr int OFF_KEEP = OFF_LD + 2 * 2 * BQ * 4;
  static constexpr int OFF_BAR = OFF_KEEP + 2 * 2 * BKV * 8;
  // kv_full, q_full[QS], q_empty[QS], sdp_full, sdp_empty, pds_full[PS], pds_empty[PS],
  // dq_full[2], dq_empty[2], ld_full[2], dkdv_full, drain[3], keep_full[4], keep_empty[4],
  // qo_full, qo_empty
  static constexpr int NBAR = 1 + 2 * QS + 1 + 1 + 2 * PS + 2 + 2 + 2 + 1 + 3 + 8 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 640;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = BQ;
  static constexpr uint32_t COL_DQ = 2 * BQ;        // DQB buffers of 64 columns
  static constexpr uint32_t COL_PT = COL_DQ + 64 * DQB;      // P^T, 16-bit pairs (PT_TMEM)
  static constexpr uint32_t COL_DST = COL_PT + BQ / 2;       // dS^T, 16-bit pairs (PT_TMEM)
  static constexpr uint32_t COL_DV = PT_TMEM ? COL_DST + BQ / 2 : COL_DQ + 128;
  static constexpr uint32_t COL_DK = COL_DV + DA;
  static_assert(COL_DK + DA <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status) {
  const bool ok = mbar_wait(bar, parity, abort, status, kStatusTimeout);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Thread-owned row of a [rows, dh] 16-bit tensor, written from TMEM columns
// [taddr, taddr + dh) times `mul` (skipped when `valid` is false); dh <= D is
// a multiple of 32.
template <int D, bool BF16>
__device__ __forceinline__ void store_rows_from_tmem(uint32_t taddr, uint4* dst, bool valid, float mul, int dh) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    if (32 * c >= dh) break;
    float v[32];
    tmem_ld32(taddr + 32 * c, v);
    tmem_ld_wait(v);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack2(v[2 * i] * mul, v[2 * i + 1] * mul, BF16);
    if (valid) {
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[4 * c + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
}

// The same rows (all 128, times `mul`) into the 128-byte-swizzled shared-memory
// slabs of a TMA store, 64 columns (128 rows x 128 bytes) per slab; `zero`
// stages zeros instead.
template <int DA, bool BF16>
__device__ __forceinline__ void stage_rows_from_tmem(uint32_t taddr, uint8_t* stage, int r, float mul, bool zero) {
#pragma unroll
  for (int c = 0; c < DA / 32; ++c) {
    uint32_t pk[16];
    if (zero) {
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = 0u;
    } else {
      float v[32];
      tmem_ld32(taddr + 32 * c, v);
      tmem_ld_wait(v);
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = pack2(v[2 * i] * mul, v[2 * i + 1] * mul, BF16);
    }
    uint8_t* slab = stage + ((32 * c) >> 6) * (128 * 128);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(slab + sw128_offset(r, (32 * c & 63) + 8 * q)) =
          make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
  }
}

// One thread of a warpgroup stores the staged 128 x DA tile (rows from key
// kv0 of head `bh`, features from feat0) with TMA; rows past Nk and features
// past dh fall outside the tensor map and are not written.
template <int DA>
__device__ __forceinline__ void store_staged_tile(const CUtensorMap* m, const uint8_t* stage, int feat0, int dh,
                                                  int2 coord) {
#pragma unroll
  for (int sl = 0; sl < DA / 64; ++sl)
    if (feat0 + 64 * sl < dh) tma_store_3d(m, stage + sl * (128 * 128), feat0 + 64 * sl, coord.x, coord.y);
  tma_store_commit();
  tma_store_wait_read();
}

template <int D, bool CAUSAL, bool BF16, bool SPARSE, bool DROP, bool VARLEN>
__global__ void __launch_bounds__(640, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                       void* __restrict__ dk, void* __restrict__ dv, const float* __restrict__ lse,
                       const float* __restrict__ delta, float* __restrict__ dq_accum, SeqLayout lay, int BH,
                       float scale, float scale_log2, const uint8_t* __restrict__ block_mask, int mask_heads,
                       DropParams drop, int group, unsigned int* status) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sP = smem + C::OFF_P;
  uint8_t* sDS = smem + C::OFF_DS;
  float* sLD = reinterpret_cast<float*>(smem + C::OFF_LD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = kv_full + 1;
  uint64_t* q_empty = q_full + C::QS;
  uint64_t* sdp_full = q_empty + C::QS;
  uint64_t* sdp_empty = sdp_full + 1;
  uint64_t* pds_full = sdp_empty + 1;
  uint64_t* pds_empty = pds_full + C::PS;
  uint64_t* dq_full = pds_empty + C::PS;
  uint64_t* dq_empty = dq_full + 2;
  uint64_t* ld_full = dq_empty + 2;
  uint64_t* dkdv_full = ld_full + 2;
  uint64_t* drain = dkdv_full + 1;
  uint64_t* keep_full = drain + 3;       // [buffer * 2 + warpgroup]
  uint64_t* keep_empty = keep_full + 4;  // [buffer * 2 + warpgroup]
  uint2* sKeep = reinterpret_cast<uint2*>(smem + C::OFF_KEEP);  // [buffer * 2 + warpgroup][key]
  uint64_t* qo_full = keep_empty + 4;   // SPLIT: the other feature half of the Q / dO stage
  uint64_t* qo_empty = qo_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heads are taken in groups of `group` (chosen by the launcher so that a
  // group's Q, dO and float32 dQ accumulators fit in about half of L2): the
  // CTAs of a group run together, and inside a group key tile 0 of every head
  // (which sees every query tile under the causal mask) goes first, then key
  // tile 1, ...: the longest CTAs start early instead of at the end.
  const int kGroup = group;
  const int n_kvt = (lay.Nk + C::BKV - 1) / C::BKV;  // key tiles of the longest sequence
  const int pass = blockIdx.x % C::NP;  // feature half (D = 256), else 0
  const int feat0 = pass * C::DA;       // first feature of dK / dV / dQ in this CTA
  const int cta = blockIdx.x / C::NP;
  const int gi = cta / (kGroup * n_kvt);
  const int heads = min(kGroup, BH - gi * kGroup);  // the last group may be smaller
  const int within = cta - gi * kGroup * n_kvt;
  const int bh = gi * kGroup + within % heads;
  const int j = within / heads;
  const int kv0 = j * C::BKV;
  const SeqView sv = seq_view<VARLEN>(lay, bh);
  if (!sv.ok && kv0 == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadSeqlens);
  if (kv0 >= sv.nk) return;  // past the end of a shorter (or rejected) sequence: the whole CTA leaves
  const int Nq = sv.nq, Nk = sv.nk;
  const int off = Nk - Nq;  // causal: key visible iff key <= query + off
  const int dh = lay.dh;
  const int n_q = (Nq + BQ - 1) / BQ;
  // Causal: the first query that sees key kv0 is kv0 - off.
  const int i_begin = CAUSAL ? (kv0 - off <= 0 ? 0 : (kv0 - off) / BQ) : 0;
  // Query tiles this key tile meets: [i_begin, n_q), and under a block mask
  // only those whose 128-row query block keeps key tile j.  Every role walks
  // the same sequence; `it` counts the tiles visited.
  const uint8_t* mcol = SPARSE ? block_mask + (long long)(mask_heads == 1 ? 0 : bh) * n_kvt * n_kvt + j : nullptr;
  auto next_tile = [&](int i) {
    if (SPARSE)
      while (i < n_q && mcol[(long long)((i * BQ) / C::BKV) * n_kvt] == 0) ++i;
    return i;
  };
  int n_it = 0;
  if (SPARSE) {
    for (int i = next_tile(i_begin); i < n_q; i = next_tile(i + 1)) ++n_it;
  } else {
    n_it = n_q > i_begin ? n_q - i_begin : 0;
  }

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int b = 0; b < C::QS; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
    }
    mbar_init(qo_full, 1);
    mbar_init(qo_empty, 2);  // the S^T and dP^T issuers
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dq_full[b], 1);
      mbar_init(&dq_empty[b], 8);
      mbar_init(&ld_full[b], 8);
    }
    mbar_init(sdp_full, 2);
    mbar_init(sdp_empty, 8);
    for (int b = 0; b < C::PS; ++b) {
      mbar_init(&pds_full[b], 8);
      mbar_init(&pds_empty[b], 2);
    }
    mbar_init(dkdv_full, 1);
    for (int i = 0; i < 3; ++i) mbar_init(&drain[i], 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&keep_full[i], 4);   // the drain warpgroup that draws them
      mbar_init(&keep_empty[i], 4);  // the compute warpgroup that uses them
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_TILE);
      const int2 ck = sv.kcoord(kv0);
      for (int s = 0; s < C::SLABS; ++s) {
        tma_load_3d(sK + s * C::KV_SLAB, &tm_k, kv_full, s * 64, ck.x, ck.y);
        tma_load_3d(sV + s * C::KV_SLAB, &tm_v, kv_full, s * 64, ck.x, ck.y);
      }
      int issued = 0, issued_o = 0;
      for (int it = 0, i = next_tile(i_begin); it < n_it; ++it, i = next_tile(i + 1)) {
        const int b = it % C::QS;
        const uint32_t use = (uint32_t)(it / C::QS);
        const int2 cq = sv.qcoord(i * BQ);
        if constexpr (C::SPLIT) {
          // the slabs outside this CTA's feature half, once S^T / dP^T of the
          // previous tile are done with them
          if (!mbar_wait(qo_empty, (use & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
          mbar_arrive_expect_tx(qo_full, 2 * (C::SLABS - C::DA / 64) * C::Q_SLAB);
          for (int s = 0; s < C::SLABS; ++s) {
            if (s / (C::DA / 64) == pass) continue;
            tma_load_3d(sQ + s * C::Q_SLAB, &tm_q, qo_full, s * 64, cq.x, cq.y);
            tma_load_3d(sDO + s * C::Q_SLAB, &tm_do, qo_full, s * 64, cq.x, cq.y);
          }
          issued_o = it + 1;
        }
        if (!mbar_wait(&q_empty[b], (use & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
        mbar_arrive_expect_tx(&q_full[b], C::SPLIT ? 2 * (C::DA / 64) * C::Q_SLAB : 2 * C::Q_TILE);
        for (int s = 0; s < C::SLABS; ++s) {
          if (C::SPLIT && s / (C::DA / 64) != pass) continue;
          tma_load_3d(sQ + b * C::Q_TILE + s * C::Q_SLAB, &tm_q, &q_full[b], s * 64, cq.x, cq.y);
          tma_load_3d(sDO + b * C::Q_TILE + s * C::Q_SLAB, &tm_do, &q_full[b], s * 64, cq.x, cq.y);
        }
        issued = it + 1;
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        drain_wait(kv_full, 0);
        for (int it = issued - C::QS < 0 ? 0 : issued - C::QS; it < issued; ++it)
          drain_wait(&q_full[it % C::QS], (uint32_t)((it / C::QS) & 1));
        if (C::SPLIT && issued_o > 0) drain_wait(qo_full, (uint32_t)((issued_o - 1) & 1));
      }
    }
  } else if (warp >= 1 && warp <= 3) {
    // ------------------------------------------------------------ MMA issuers
    // A single thread issues at most one tcgen05.mma every ~100 cycles, so
    // the five products are spread over three issuing threads:
    //   warp 1: S^T(i+1) = K Q^T, then the dQ partial of tile i
    //   warp 2: dP^T(i+1) = V dO^T
    //   warp 3: dV += P^T dO, dK += dS^T Q of tile i
    if (lane == 0) {
      constexpr uint32_t kIdSdP = idesc_f16(128, BQ, BF16, false, false);   // K-major A, K-major B
      constexpr uint32_t kIdAcc = idesc_f16(128, C::DA, BF16, false, true);  // K-major A, MN-major B
      constexpr uint32_t kIdDq = idesc_f16(128, 64, BF16, true, true);      // MN-major A and B
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO);
      const uint32_t aP = smem_u32(sP), aDS = smem_u32(sDS);
      // S^T = K Q^T (warp 1) or dP^T = V dO^T (warp 2) for the tile in stage qs.
      // SPLIT: the K steps over the other feature half (its slabs arrive
      // first; the first of them starts the accumulator), then those over
      // this CTA's half.
      constexpr int kHalfSteps = C::DA / 16;
      const int kk_other = pass == 0 ? kHalfSteps : 0;
      const int kk_own = pass == 0 ? 0 : kHalfSteps;
      auto issue_sdp_half = [&](int kk0, bool start) {
        const uint64_t da = sdesc_sw128(warp == 1 ? aK : aV, 16, 1024);
        const uint64_t db = sdesc_sw128(warp == 1 ? aQ : aDO, 16, 1024);
        const uint32_t dcol = tmem + (warp == 1 ? C::COL_S : C::COL_DP);
#pragma unroll
        for (int t = 0; t < kHalfSteps; ++t) {
          const int kk = kk0 + t;
          const uint32_t ok = ((kk >> 2) * C::KV_SLAB + (kk & 3) * 32) >> 4;
          const uint32_t oq = ((kk >> 2) * C::Q_SLAB + (kk & 3) * 32) >> 4;
          mma_ss(dcol, da + ok, db + oq, kIdSdP, !(start && t == 0));
        }
      };
      auto issue_sdp = [&](int qs) {
        const uint64_t da = sdesc_sw128(warp == 1 ? aK : aV, 16, 1024);
        const uint64_t db = sdesc_sw128((warp == 1 ? aQ : aDO) + qs * C::Q_TILE, 16, 1024);
        const uint32_t dcol = tmem + (warp == 1 ? C::COL_S : C::COL_DP);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ok = ((kk >> 2) * C::KV_SLAB + (kk & 3) * 32) >> 4;
          const uint32_t oq = ((kk >> 2) * C::Q_SLAB + (kk & 3) * 32) >> 4;
          mma_ss(dcol, da + ok, db + oq, kIdSdP, kk > 0);
        }
      };
      // dV += P^T dO and dK += dS^T Q (warp 3); A from TMEM when PT_TMEM.
      auto issue_dkdv = [&](int qs, int pb, bool first) {
        const uint64_t dp = sdesc_sw128(aP + pb * C::PT_TILE, 16, 1024);
        const uint64_t dds = sdesc_sw128(aDS + pb * C::PT_TILE, 16, 1024);
        // this CTA's feature half: slabs feat0 / 64 ..
        const uint32_t fo = (feat0 / 64) * C::Q_SLAB;
        const uint64_t ddo = sdesc_sw128(aDO + qs * C::Q_TILE + fo, C::Q_SLAB, 1024);
        const uint64_t dq = sdesc_sw128(aQ + qs * C::Q_TILE + fo, C::Q_SLAB, 1024);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t op = ((kk >> 2) * C::PT_SLAB + (kk & 3) * 32) >> 4;
          if (C::PT_TMEM)
            mma_ts(tmem + C::COL_DV, tmem + C::COL_PT + kk * 8, ddo + ((kk * 2048) >> 4), kIdAcc, !(first && kk == 0));
          else
            mma_ss(tmem + C::COL_DV, dp + op, ddo + ((kk * 2048) >> 4), kIdAcc, !(first && kk == 0));
        }
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t op = ((kk >> 2) * C::PT_SLAB + (kk & 3) * 32) >> 4;
          if (C::PT_TMEM)
            mma_ts(tmem + C::COL_DK, tmem + C::COL_DST + kk * 8, dq + ((kk * 2048) >> 4), kIdAcc, !(first && kk == 0));
          else
            mma_ss(tmem + C::COL_DK, dds + op, dq + ((kk * 2048) >> 4), kIdAcc, !(first && kk == 0));
        }
      };
      // dQ partial -> TMEM buffer b (warp 1).
      auto issue_dq = [&](int pb, int b) {
        const uint64_t dk0 = sdesc_sw128(aK + (feat0 / 64) * C::KV_SLAB, C::KV_SLAB, 1024);
        const uint64_t ds0 = sdesc_sw128(aDS + pb * C::PT_TILE, C::PT_SLAB, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BKV / 16; ++kk) {
          const uint32_t o = (kk * 2048) >> 4;
          if (C::DQT)  // dQ^T = K^T dS^T
            mma_ss(tmem + C::COL_DQ + 64 * b, dk0 + o, ds0 + o, kIdDq, kk > 0);
          else         // dQ = dS K
            mma_ss(tmem + C::COL_DQ + 64 * b, ds0 + o, dk0 + o, kIdDq, kk > 0);
        }
      };
      // SPLIT: S^T / dP^T of tile t over the other feature half (then that
      // half of the stage is released), and over this CTA's half.
      auto sdp_other = [&](int t) {
        if (!mbar_wait(qo_full, t & 1, abort_flag, status, kStatusTimeout)) return false;
        tc_fence_after();
        issue_sdp_half(kk_other, true);
        mma_commit(qo_empty);
        return true;
      };
      auto sdp_own = [&](int t) {
        if (!mbar_wait(&q_full[0], t & 1, abort_flag, status, kStatusTimeout)) return false;
        tc_fence_after();
        issue_sdp_half(kk_own, false);
        mma_commit(sdp_full);
        return true;
      };
      bool ok = mbar_wait(kv_full, 0, abort_flag, status, kStatusTimeout);
      if (warp <= 2 && n_it > 0) {
        if constexpr (C::SPLIT) {
          ok = ok && sdp_other(0) && sdp_own(0);
        } else {
          if (ok) ok = mbar_wait(&q_full[0], 0, abort_flag, status, kStatusTimeout);
          if (ok) {
            tc_fence_after();
            issue_sdp(0);
            mma_commit(sdp_full);
          }
        }
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int b = it % C::DQB;
        const int qs = it % C::QS;
        const int pb = it % C::PS;
        if (warp <= 2 && it + 1 < n_it) {
          const int qn = (it + 1) % C::QS;
          if (!(ok = mbar_wait(sdp_empty, it & 1, abort_flag, status, kStatusTimeout))) break;
          if constexpr (C::SPLIT) {
            // warp 1 issues its own half after the dQ product of tile it
            if (!(ok = sdp_other(it + 1))) break;
            if (warp == 2 && !(ok = sdp_own(it + 1))) break;
          } else {
            if (!(ok = mbar_wait(&q_full[qn], ((it + 1) / C::QS) & 1, abort_flag, status, kStatusTimeout))) break;
            tc_fence_after();
            issue_sdp(qn);
            mma_commit(sdp_full);
          }
        }
        if (warp == 2) continue;
        if (!(ok = mbar_wait(&pds_full[pb], (it / C::PS) & 1, abort_flag, status, kStatusTimeout))) break;
        if (warp == 1) {
          if (!(ok = mbar_wait(&dq_empty[b], ((it / C::DQB) & 1) ^ 1, abort_flag, status, kStatusTimeout))) break;
          tc_fence_after();
          issue_dq(pb, b);
          mma_commit(&dq_full[b]);
          mma_commit(&pds_empty[pb]);
          if constexpr (C::SPLIT) {
            if (it + 1 < n_it && !(ok = sdp_own(it + 1))) break;
          }
        } else {
          tc_fence_after();
          issue_dkdv(qs, pb, it == 0);
          mma_commit(&pds_empty[pb]);
          mma_commit(&q_empty[qs]);
        }
      }
      if (ok && warp == 3) {
        mma_commit(dkdv_full);
        // score blocks of this key tile (counted once, by feature half 0)
        if (pass == 0) count_score_blocks(status, kCountBackward, (unsigned long long)n_it * (C::BKV / 64) * (BQ / 64));
      }
      if (!ok) {  // every MMA this thread issued must finish before TMEM is freed
        mma_commit(&drain[warp - 1]);
        drain_wait(&drain[warp - 1], 0);
      }
    }
  } else if ((warp >= 4 && warp < 8) || (warp >= 12 && warp < 16)) {
    // ------------------------------------------------------------ compute: P^T, dS^T
    // Warpgroup h = 0 (warps 4-7) owns query columns [0, CW) of every tile,
    // h = 1 (warps 12-15) owns [CW, BQ); one key row per thread (TMEM lane),
    // 16 columns at a time.
    constexpr int CW = BQ / 2;
    const int h = warp >= 12 ? 1 : 0;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int key = kv0 + r;
    const int key_rel = key - off;  // causal: masked iff key_rel > query
    const int kv0_rel = kv0 - off;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    // Per query column: -LSE*log2(e) (so that P = exp2(s*scale*log2e - LSE*log2e))
    // and -D, staged in shared memory one iteration ahead.
    float pre_l = 0.f, pre_d = 0.f;
    auto fetch = [&](int i) {  // query tile i
      const int q = i * BQ + h * CW + r;
      if (r < CW) {
        if (q < Nq) {
          const float lq = lse[sv.qflat(q)];
          pre_l = lq == -pos_inf() ? -pos_inf() : -lq * kLog2e;  // a row with no visible key: P = 0
          pre_d = -delta[sv.qflat(q)];
        } else {  // padding query: P = exp2(-inf) = 0
          pre_l = -pos_inf();
          pre_d = 0.f;
        }
      }
    };
    // Dropout keep bits of this thread's key for the CW query columns of the
    // current tile (bit c of kw0 <-> query column c of this warpgroup, bit c
    // of kw1 <-> column 32 + c), drawn one tile ahead by the dQ drain warps of
    // the same TMEM lanes (key_keep_words in fa_philox.cuh).
    uint32_t kw0 = 0u, kw1 = 0u;
    int i = next_tile(i_begin);
    fetch(i);
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int lb = it & 1;
      const int pb = it % C::PS;
      float* sNL = sLD + lb * 2 * BQ;
      float* sND = sNL + BQ;
      if (r < CW) {
        sNL[h * CW + r] = pre_l;
        sND[h * CW + r] = pre_d;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ld_full[lb]);
      if (!(ok = warp_wait(&ld_full[lb], (it >> 1) & 1, abort_flag, status))) break;
      const int q0 = i * BQ;
      i = next_tile(i + 1);
      if (it + 1 < n_it) fetch(i);
      if (!(ok = warp_wait(sdp_full, it & 1, abort_flag, status))) break;
      if (DROP) {
        const int kb = (it & 1) * 2 + h;
        if (!(ok = warp_wait(&keep_full[kb], (it >> 1) & 1, abort_flag, status))) break;
        const uint2 kw = sKeep[kb * C::BKV + r];
        kw0 = kw.x;
        kw1 = kw.y;
        __syncwarp();
        if (lane == 0) mbar_arrive(&keep_empty[kb]);
      }
      tc_fence_after();
#pragma unroll 1
      for (int sc = 0; sc < CW / 16; ++sc) {
        const int col = h * CW + 16 * sc;  // first column of this 16-column sub-chunk
        float s[16], dp[16];
        tmem_ld16(lane_base + C::COL_S + col, s);
        tmem_ld16(lane_base + C::COL_DP + col, dp);
        tmem_ld_wait(s);
        tmem_ld_wait(dp);
        if (sc == CW / 16 - 1) {  // S^T / dP^T columns may now be overwritten by the next tile
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sdp_empty);
        }
        const int c0 = q0 + col;  // first query of this sub-chunk
        const bool need_mask = (CAUSAL && c0 < kv0_rel + C::BKV - 1) || (kv0 + C::BKV > Nk);
        const uint32_t keep = DROP ? (((sc >> 1) ? kw1 : kw0) >> (16 * (sc & 1))) : 0xffffu;  // bit c: (c0 + c, key) kept
        uint32_t pp[8], dd[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = 2 * i;
          const float2 nl = *reinterpret_cast<const float2*>(sNL + col + c);
          const float2 nd = *reinterpret_cast<const float2*>(sND + col + c);
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sc2, f2_pack(nl.x, nl.y)), x0, x1);
          float p0 = ex2_approx(x0);
          float p1 = ex2_approx(x1);
          if (need_mask) {
            if (key >= Nk || (CAUSAL && key_rel > c0 + c)) p0 = 0.f;
            if (key >= Nk || (CAUSAL && key_rel > c0 + c + 1)) p1 = 0.f;
          }
          float dp0 = dp[c], dp1 = dp[c + 1];
          float pv0 = p0, pv1 = p1;  // dV operand: the kept P
          if (DROP) {
            const bool k0 = (keep >> c) & 1u, k1 = (keep >> (c + 1)) & 1u;
            dp0 = k0 ? dp0 * drop.keep_scale : 0.f;
            dp1 = k1 ? dp1 * drop.keep_scale : 0.f;
            pv0 = k0 ? p0 : 0.f;
            pv1 = k1 ? p1 : 0.f;
          }
          const uint64_t t2 = f2_add(f2_pack(dp0, dp1), f2_pack(nd.x, nd.y));
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p0, p1), t2), d0, d1);
          pp[i] = pack2(pv0, pv1, BF16);
          dd[i] = pack2(d0, d1, BF16);
        }
        // The buffers are free once the products of the previous tile are done.
        if (sc == 0 && !(ok = warp_wait(&pds_empty[pb], ((it / C::PS) & 1) ^ 1, abort_flag, status))) break;
        if (C::PT_TMEM) {
          tmem_st8(lane_base + C::COL_PT + col / 2, pp);
          tmem_st8(lane_base + C::COL_DST + col / 2, dd);
        } else {
          uint8_t* prow = sP + pb * C::PT_TILE + (col >> 6) * C::PT_SLAB;
#pragma unroll
          for (int q = 0; q < 2; ++q)
            *reinterpret_cast<uint4*>(prow + sw128_offset(r, (col & 63) + 8 * q)) =
                make_uint4(pp[4 * q], pp[4 * q + 1], pp[4 * q + 2], pp[4 * q + 3]);
        }
        uint8_t* drow = sDS + pb * C::PT_TILE + (col >> 6) * C::PT_SLAB;
#pragma unroll
        for (int q = 0; q < 2; ++q)
          *reinterpret_cast<uint4*>(drow + sw128_offset(r, (col & 63) + 8 * q)) =
              make_uint4(dd[4 * q], dd[4 * q + 1], dd[4 * q + 2], dd[4 * q + 3]);
      }
      if (!ok) break;
      if (C::PT_TMEM) tmem_st_wait();
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pds_full[pb]);
    }
    if (h == 0) {
      if (ok) ok = warp_wait(dkdv_full, 0, abort_flag, status);
      if (ok) tc_fence_after();
      // n_it == 0: no query sees this key tile (block mask, or causal with Nq < Nk): dV = 0
      if constexpr (!VARLEN) {
        // Dense rows: stage the tile in the (now unused) Q stages, store with
        // TMA; every warp of the warpgroup reaches the barrier once.
        if (ok) stage_rows_from_tmem<C::DA, BF16>(lane_base + C::COL_DV, sQ, r, DROP ? drop.keep_scale : 1.f,
                                                  n_it == 0);
        fence_async_smem();
        named_barrier_sync(1, 128);
        if (r == 0 && ok && !*abort_flag) store_staged_tile<C::DA>(&tm_dv, sQ, feat0, dh, sv.kcoord(kv0));
      } else if (ok) {
        uint4* dst = reinterpret_cast<uint4*>(dv) + sv.kflat(key) * (dh / 8) + feat0 / 8;
        const int cols = min(C::DA, dh - feat0);  // features of this CTA that exist
        if (n_it > 0) {
          store_rows_from_tmem<C::DA, BF16>(lane_base + C::COL_DV, dst, key < Nk, DROP ? drop.keep_scale : 1.f,
                                            cols);
        } else if (key < Nk) {
          for (int q = 0; q < cols / 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
  } else if ((warp >= 8 && warp < 12) || warp >= 16) {
    // ------------------------------------------------------------ dQ drain
    // Two warpgroups (g = 0: warps 8-11, g = 1: warps 16-19) each add 32 of
    // the 64 columns of the dQ partial into the float32 accumulator.
    const int g = warp >= 16 ? 1 : 0;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = true;
    // Dropout keep words of tile `it` (query tile i) for compute warpgroup g:
    // drawn here, one tile ahead, where the drain warps would otherwise wait.
    auto draw = [&](int it, int i) {
      const int kb = (it & 1) * 2 + g;
      if (!warp_wait(&keep_empty[kb], ((it >> 1) & 1) ^ 1, abort_flag, status)) return false;
      sKeep[kb * C::BKV + r] = key_keep_words(kv0 + r, i * BQ + g * (BQ / 2), BQ / 2, lane, bh, drop);
      __syncwarp();
      if (lane == 0) mbar_arrive(&keep_full[kb]);
      return true;
    };
    if (DROP && n_it > 0) ok = draw(0, next_tile(i_begin));
    for (int it = 0, i = next_tile(i_begin); ok && it < n_it; ++it, i = next_tile(i + 1)) {
      const int b = it % C::DQB;
      if (DROP && it + 1 < n_it && !(ok = draw(it + 1, next_tile(i + 1)))) break;
      if (!(ok = warp_wait(&dq_full[b], (it / C::DQB) & 1, abort_flag, status))) break;
      tc_fence_after();
      float v[32];
      tmem_ld32(lane_base + C::COL_DQ + 64 * b + 32 * g, v);
      tmem_ld_wait(v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dq_empty[b]);
      const int q0 = i * BQ;
      if (C::DQT) {  // lane = feature r, column = query q0 + 32g + c: one 128-byte line per warp and column
        float* base = dq_accum + sv.qflat(q0 + 32 * g) * dh + feat0 + r;
        if (!sv.varlen && dh == D) {  // dense rows D floats apart: constant offsets
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (q0 + 32 * g + c < Nq) red_add_f32(base + c * D, v[c]);
        } else if (feat0 + r < dh) {
          const long long step = (long long)sv.rstride * dh;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (q0 + 32 * g + c < Nq) red_add_f32(base + c * step, v[c]);
        }
      } else {  // lane = query q0 + r, column = feature 32g + c (dh = D = 64)
        if (q0 + r < Nq) {
          float* base = dq_accum + sv.qflat(q0 + r) * dh + 32 * g;
#pragma unroll
          for (int c = 0; c < 32; c += 4) red_add_v4(base + c, v[c], v[c + 1], v[c + 2], v[c + 3]);
        }
      }
    }
    if (g == 0) {
      if (ok) ok = warp_wait(dkdv_full, 0, abort_flag, status);
      if (ok) tc_fence_after();
      if constexpr (!VARLEN) {  // as dV, staged in the dO stages
        if (ok) stage_rows_from_tmem<C::DA, BF16>(lane_base + C::COL_DK, sDO, r, scale, n_it == 0);
        fence_async_smem();
        named_barrier_sync(2, 128);
        if (r == 0 && ok && !*abort_flag) store_staged_tile<C::DA>(&tm_dk, sDO, feat0, dh, sv.kcoord(kv0));
      } else if (ok) {
        const int key = kv0 + r;
        uint4* dst = reinterpret_cast<uint4*>(dk) + sv.kflat(key) * (dh / 8) + feat0 / 8;
        const int cols = min(C::DA, dh - feat0);
        if (n_it > 0) {
          store_rows_from_tmem<C::DA, BF16>(lane_base + C::COL_DK, dst, key < Nk, scale, cols);
        } else if (key < Nk) {  // dK = 0 likewise
          for (int q = 0; q < cols / 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
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

// Heads per CTA group: Q and dO (16-bit) and the float32 dQ accumulator of a
// head take 8 * Nq * d bytes; a group keeps them within ~64 MB of L2.
inline int heads_per_group(const BwdArgs& a, int D) {
  const long long per_head = 8LL * a.lay.Nq * D;
  long long g = (64LL << 20) / (per_head > 0 ? per_head : 1);
  if (g > 16) g = 16;
  if (g < 1) g = 1;
  return (int)g;
}

template <int D, bool CAUSAL, bool BF16, bool SPARSE, bool DROP, bool VARLEN>
cudaError_t launch_dkdv_t(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kern = fa_bwd_dkdv_kernel<D, CAUSAL, BF16, SPARSE, DROP, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_kv = (a.lay.Nk + C::BKV - 1) / C::BKV;
  const long long grid = (long long)n_kv * a.BH * C::NP;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_do, a.tm_k, a.tm_v, a.tm_dk, a.tm_dv, a.dk,
                                                         a.dv, a.lse,
                                                         a.delta, a.dq_accum, a.lay, a.BH, a.scale, a.scale_log2,
                                                         a.block_mask, a.mask_heads, a.drop, heads_per_group(a, D),
                                                         a.status);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fa

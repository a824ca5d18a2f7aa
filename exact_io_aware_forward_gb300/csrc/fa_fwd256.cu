// Forward pass at head dimension 256 on sm_103a.
//
// Same recurrence as fa_fwd_kernel.cuh ("FlashAttention 为什么不需要存下注意力矩阵",
// jefxiong.cn, section 3.2): running max m, sum l and unnormalised O per
// query row, rescaled lazily; only O and LSE = m + ln l leave the chip.
//
// Why a separate kernel: at d = 256 one 128 x 256 fp32 O accumulator takes
// 256 of the 512 TMEM columns, so the two ping-ponging query tiles of the
// d <= 128 kernel (2 x S + 2 x O = 768 columns) do not fit.  Here a CTA owns
// ONE 128-row query tile and overlaps its own softmax with the tensor core by
// double-buffering S:
//   TMEM  S_a (128 cols) | S_b (128 cols) | O (256 cols)
//   MMA order  S(0) S(1) | PV(0) S(2) | PV(1) S(3) | ...
// so the tensor core computes PV(j) and S(j+2) while the softmax warps work on
// S(j+1).  Key tiles are 128 keys, so every product is a 128 x 128 x 16
// instruction: S over 16 K-steps of the 256 features, and PV as two N = 128
// products, one per 128-feature half of V and O (64-key tiles, which made
// the S products N = 64, cost nearly as much per instruction for half the
// work).  K and V move through the ring in 128-feature halves (32 KB slots),
// so that Q (64 KB) and five slots fit in shared memory.
//
// Roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: Q once, then K / V half tiles in consumption
//               order K0 K1 V0 K2 V1 K3 V2 ... (each as its two feature
//               halves) through a 5-slot ring.
//   warp 1      TMEM allocation; lane 0 issues every tcgen05.mma.
//   warps 2-5   softmax, one query row per thread (TMEM lane), then the
//               epilogue (O / l_mma, LSE).
// PV(j-1) can still be accumulating into O while the softmax of tile j runs,
// so a row that needs its O rescaled first waits for the commit of PV(j-1).
#include "fa_fwd_kernel.cuh"

namespace fa {
namespace {

struct Fwd256Cfg {
  static constexpr int D = 256;
  static constexpr int BM = 128;                   // query rows per CTA
  static constexpr int BN = 128;                   // keys per tile
  static constexpr int Q_SLAB = 128 * 64 * 2;      // 128 rows x 64 features x 16 bit
  static constexpr int KV_SLAB = 128 * 64 * 2;     // 128 keys x 64 features
  static constexpr int SLABS = D / 64;
  static constexpr int Q_TILE = SLABS * Q_SLAB;    // 64 KB
  static constexpr int KV_TILE = 2 * KV_SLAB;      // one ring slot: 128 keys x 128 features, 32 KB
  static constexpr int NS = 5;                     // ring slots
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = Q_TILE;
  static constexpr int OFF_BAR = OFF_RING + NS * KV_TILE;
  // q_full, ring_full[NS], ring_empty[NS], s_full[2], p_full[2], pv_done, o_full, drain
  static constexpr int NBAR = 1 + 2 * NS + 2 + 2 + 1 + 1 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;    // S_a at 0, S_b at 128
  static constexpr uint32_t COL_O = 256;  // 256 columns
  static_assert(SMEM <= 232448, "shared memory budget");
};

// The ring carries K and V tiles in the order the MMA thread consumes them:
// K0, K1, then V(j), K(j+2) for j = 0, 1, ... (K(j+2) only while it exists),
// each as two consecutive positions (feature halves).  Tile position p of
// that sequence -> (is_v, tile).
__device__ __forceinline__ void ring_item(int p, int n, bool& is_v, int& tile) {
  if (p < 2 && p < n) {
    is_v = false;
    tile = p;
    return;
  }
  const int first = n < 2 ? n : 2;  // K tiles before the first V
  const int q = p - first;
  // After the prefix: V0, K2, V1, K3, ... while K(j+2) < n; then only V's.
  const int pairs = n - 2 > 0 ? n - 2 : 0;  // number of K(j+2) entries
  if (q < 2 * pairs) {
    is_v = (q & 1) == 0;
    tile = is_v ? q / 2 : q / 2 + 2;
  } else {
    is_v = true;
    tile = pairs + (q - 2 * pairs);
  }
}

template <bool CAUSAL, bool BF16, bool DROP, bool VARLEN>
__global__ void __launch_bounds__(192, 1)
    fa_fwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, void* __restrict__ o, float* __restrict__ lse,
                     SeqLayout lay, int BH, int n_qblocks, float scale_log2, DropParams drop, int group,
                     unsigned int* status) {
  using C = Fwd256Cfg;
  constexpr int D = C::D;
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
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_full = pv_done + 1;
  uint64_t* drain = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heads in groups of `group` (a group's K and V fit in about half of L2, so
  // they are read from DRAM about once); inside a group the heaviest work
  // first: under the causal mask the last query blocks see the most keys.
  const int gi = blockIdx.x / (group * n_qblocks);
  const int heads = min(group, BH - gi * group);  // the last group may be smaller
  const int within = blockIdx.x - gi * group * n_qblocks;
  const int bh = gi * group + within % heads;
  const int qb = n_qblocks - 1 - within / heads;
  const int q0 = qb * C::BM;
  const SeqView sv = seq_view<VARLEN>(lay, bh);
  if (!sv.ok && q0 == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadSeqlens);
  if (q0 >= sv.nq) return;  // past the end of a shorter (or rejected) sequence
  const int Nq = sv.nq, Nk = sv.nk;
  const int off = Nk - Nq;  // causal: key visible iff key <= row + off
  const int n_kv = (Nk + C::BN - 1) / C::BN;
  const int n = CAUSAL ? causal_key_tiles(q0 + C::BM - 1, off, n_kv, C::BN) : n_kv;  // key tiles visited
  const int n_items = 4 * n;  // ring positions: both halves of every K and every V once

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
    }
    mbar_init(pv_done, 1);
    mbar_init(o_full, 1);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(q_full, C::Q_TILE);
      const int2 cq = sv.qcoord(q0);
      for (int s = 0; s < C::SLABS; ++s) tma_load_3d(sQ + s * C::Q_SLAB, &tm_q, q_full, s * 64, cq.x, cq.y);
      for (int p = 0; p < n_items; ++p) {
        const int slot = p % C::NS;
        const uint32_t use = (uint32_t)(p / C::NS);
        if (!mbar_wait(&ring_empty[slot], (use & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
        bool is_v;
        int tile;
        ring_item(p >> 1, n, is_v, tile);
        const int half = p & 1;  // features [128 half, 128 half + 128)
        mbar_arrive_expect_tx(&ring_full[slot], C::KV_TILE);
        const int2 ck = sv.kcoord(tile * C::BN);
        for (int s = 0; s < 2; ++s)
          tma_load_3d(sRing + slot * C::KV_TILE + s * C::KV_SLAB, is_v ? &tm_v : &tm_k, &ring_full[slot],
                      128 * half + 64 * s, ck.x, ck.y);
        issued = p + 1;
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        drain_wait(q_full, 0);
        for (int p = issued - C::NS < 0 ? 0 : issued - C::NS; p < issued; ++p)
          drain_wait(&ring_full[p % C::NS], (uint32_t)((p / C::NS) & 1));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, C::BN, BF16, false, false);  // K-major A and B
      constexpr uint32_t kIdPV = idesc_f16(128, 128, BF16, false, true);    // B (V) MN-major, one feature half
      const uint32_t sq = smem_u32(sQ);
      const uint32_t sring = smem_u32(sRing);
      // descriptors of Q and of ring slot 0 (K: K-major; V: MN-major), advanced per K-step
      const uint64_t dq = sdesc_sw128(sq, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sring, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sring, C::KV_SLAB, 1024);
      int pos = 0;  // next ring position to consume
      // S(j) = Q K(j)^T into S buffer b: 16 k-steps of 16 features, the first
      // 8 from K's half in ring slot k0, the last 8 from slot k1.
      auto issue_s = [&](int b, int k0, int k1) {
        const uint64_t dka = sdesc_advance(dk0, k0 * C::KV_TILE);
        const uint64_t dkb = sdesc_advance(dk0, k1 * C::KV_TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::Q_SLAB + (kk & 3) * 32;
          const uint32_t ob = ((kk >> 2) & 1) * C::KV_SLAB + (kk & 3) * 32;
          mma_ss(tmem + C::COL_S + 128 * b, sdesc_advance(dq, oa), sdesc_advance(kk < 8 ? dka : dkb, ob), kIdS,
                 kk > 0);
        }
      };
      // O += P(j) V(j): P read from S buffer b (16-bit pairs, 8 columns per 16
      // keys); O's feature half h from V's half in ring slot v_h.
      auto issue_pv = [&](int b, int v0, int v1, bool first) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t dv = sdesc_advance(dv0, (h ? v1 : v0) * C::KV_TILE);
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            mma_ts(tmem + C::COL_O + 128 * h, tmem + C::COL_S + 128 * b + kk * 8, sdesc_advance(dv, kk * 2048),
                   kIdPV, !first || kk > 0);
        }
      };
      auto take = [&](bool& ok) {  // wait for the next ring position; returns its slot
        const int slot = pos % C::NS;
        ok = mbar_wait(&ring_full[slot], (uint32_t)((pos / C::NS) & 1), abort_flag, status, kStatusTimeout);
        ++pos;
        return slot;
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, status, kStatusTimeout);
      for (int j = 0; ok && j < n && j < 2; ++j) {  // S(0), S(1)
        const int k0 = take(ok);
        const int k1 = ok ? take(ok) : 0;
        if (!ok) break;
        tc_fence_after();
        issue_s(j, k0, k1);
        mma_commit(&s_full[j]);
        mma_commit(&ring_empty[k0]);
        mma_commit(&ring_empty[k1]);
      }
      for (int j = 0; ok && j < n; ++j) {
        const int b = j & 1;
        if (!(ok = mbar_wait(&p_full[b], (uint32_t)((j >> 1) & 1), abort_flag, status, kStatusTimeout))) break;
        const int v0 = take(ok);
        const int v1 = ok ? take(ok) : 0;
        if (!ok) break;
        tc_fence_after();
        issue_pv(b, v0, v1, j == 0);
        mma_commit(&ring_empty[v0]);
        mma_commit(&ring_empty[v1]);
        mma_commit(pv_done);
        if (j + 2 < n) {  // S(j+2) reuses buffer b: in-order after PV(j), which reads P(j) there
          const int k0 = take(ok);
          const int k1 = ok ? take(ok) : 0;
          if (!ok) break;
          tc_fence_after();
          issue_s(b, k0, k1);
          mma_commit(&s_full[b]);
          mma_commit(&ring_empty[k0]);
          mma_commit(&ring_empty[k1]);
        }
      }
      mma_commit(ok ? o_full : drain);  // with no key tile this arrives at once
      if (ok) count_score_blocks(status, kCountForward, (unsigned long long)n * (C::BN / 32));  // 128 x BN each
      if (!ok) drain_wait(drain, 0);    // every MMA issued must finish before TMEM is freed
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;                 // warps 2-5 -> TMEM lanes 64-95, 96-127, 0-31, 32-63
    const int r = quarter * 32 + lane;            // row within the tile == TMEM lane
    const int row = q0 + r;
    const int row_off = row + off;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tO = lane_base + C::COL_O;

    float m_ref = neg_inf();
    float l = 0.f;
    float l_mma = 0.f;
    bool ok = true;
    uint32_t keep[4] = {0u, 0u, 0u, 0u};  // dropout bits of the next tile, 32 keys per word
    auto draw = [&](int j) { tile_keep_bits<4>(keep, j * C::BN, row, bh, drop.offset, drop.k0, drop.k1, drop.t); };
    if (DROP && n > 0) draw(0);
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      const uint32_t tS = lane_base + C::COL_S + 128 * b;
      if (!(ok = warp_wait(&s_full[b], (uint32_t)((j >> 1) & 1), abort_flag, status))) break;
      tc_fence_after();
      float s[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + 32 * cc, s[cc]);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(s[cc]);
      const int kbase = j * C::BN;
      const bool need_mask = (kbase + C::BN > Nk) || (CAUSAL && kbase + C::BN - 1 > q0 + off);
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
        rescale_o = j > 0;
        m_ref = m_use;
      }
      const float neg_m = (m_ref == neg_inf()) ? 0.f : -m_ref;
      const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
      const uint64_t nm2 = f2_pack(neg_m, neg_m);
      uint64_t sum2 = f2_pack(0.f, 0.f);
      uint64_t sumr2 = f2_pack(0.f, 0.f);
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
        // PV(j-1) may still be adding into O: wait for its commit first.
        if (!(ok = warp_wait(pv_done, (uint32_t)((j - 1) & 1), abort_flag, status))) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          float ov[32];
          tmem_ld32(tO + 32 * cc, ov);
          tmem_ld_wait(ov);
          const uint64_t corr2 = f2_pack(corr, corr);
          uint32_t ou[32];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float a, bb;
            f2_unpack(f2_mul(f2_pack(ov[i], ov[i + 1]), corr2), a, bb);
            ou[i] = __float_as_uint(a);
            ou[i + 1] = __float_as_uint(bb);
          }
          tmem_st32(tO + 32 * cc, ou);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
      if (DROP && j + 1 < n) draw(j + 1);
      float a, bb;
      f2_unpack(sum2, a, bb);
      l += a + bb;
      f2_unpack(sumr2, a, bb);
      l_mma += a + bb;
    }

    // ------------------------------------------------------------ epilogue
    if (ok) ok = warp_wait(o_full, 0, abort_flag, status);
    const long long frow = sv.qflat(row);
    if (ok) {
      tc_fence_after();
      // n = 0 (no key) or a row that saw no key: O = 0 (never accumulated / all P = 0), LSE = -inf.
      const float inv_l = (n > 0 && l_mma > 0.f) ? (DROP ? drop.keep_scale : 1.f) / l_mma : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(o) + frow * (D / 8);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        float ov[32];
        if (n > 0) {
          tmem_ld32(tO + 32 * cc, ov);
          tmem_ld_wait(ov);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0.f;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2(ov[2 * i] * inv_l, ov[2 * i + 1] * inv_l, BF16);
        if (row < Nq) {
#pragma unroll
          for (int q = 0; q < 4; ++q) orow[4 * cc + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (row < Nq) {
        const float m_fin = (m_ref == neg_inf()) ? 0.f : m_ref;
        lse[frow] = (n > 0) ? (m_fin + __log2f(l)) * kLn2 : neg_inf();
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

template <bool CAUSAL, bool BF16, bool DROP, bool VARLEN>
cudaError_t launch_fwd256_t(const FwdArgs& a, cudaStream_t stream) {
  using C = Fwd256Cfg;
  auto kern = fa_fwd256_kernel<CAUSAL, BF16, DROP, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qblocks = (a.lay.Nq + C::BM - 1) / C::BM;
  const long long grid = (long long)n_qblocks * a.BH;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // K and V of a head take 4 * Nk * 256 bytes; a group keeps them within ~64 MB of L2.
  const long long per_head = 4LL * a.lay.Nk * C::D;
  const int group = (int)std::max(1LL, std::min(64LL, (64LL << 20) / (per_head > 0 ? per_head : 1)));
  kern<<<(unsigned)grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.o, a.lse, a.lay, a.BH, n_qblocks,
                                                         a.scale_log2, a.drop, group, a.status);
  return cudaGetLastError();
}

template <bool CAUSAL, bool BF16>
cudaError_t launch_fwd256_c(const FwdArgs& a, cudaStream_t stream) {
  const bool varlen = a.lay.cu_q != nullptr;
  if (varlen)
    return a.dropout ? launch_fwd256_t<CAUSAL, BF16, true, true>(a, stream)
                     : launch_fwd256_t<CAUSAL, BF16, false, true>(a, stream);
  return a.dropout ? launch_fwd256_t<CAUSAL, BF16, true, false>(a, stream)
                   : launch_fwd256_t<CAUSAL, BF16, false, false>(a, stream);
}

}  // namespace

cudaError_t launch_forward256(bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream) {
  if (causal && bf16) return launch_fwd256_c<true, true>(a, stream);
  if (causal) return launch_fwd256_c<true, false>(a, stream);
  if (bf16) return launch_fwd256_c<false, true>(a, stream);
  return launch_fwd256_c<false, false>(a, stream);
}

}  // namespace fa

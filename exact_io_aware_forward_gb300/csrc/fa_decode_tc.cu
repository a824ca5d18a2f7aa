// Split-KV forward on the tensor cores for decoding (few queries against many
// keys), d in {64, 128, 256}: from one query per head up to several
// (speculative or chunked decoding, grouped-query heads), 128 queries per CTA.
//
// The key range of every head is cut into contiguous chunks (the plan and the
// combine kernel that merges the chunks are in fa_decode.cu); a CTA takes up
// to 128 queries of one head against one
// chunk, so each K and V tile is read from memory once for all of them,
// and evaluates the online-softmax recurrence ("FlashAttention 为什么不需要存下
// 注意力矩阵", jefxiong.cn, section 3.2) over the chunk's 128-key tiles:
//   S(j) = Q K_j^T and O += P(j) V_j on the tensor core (TMEM accumulators),
//   S double-buffered (S_a | S_b | O), in the order S(0) S(1) | PV(0) S(2) |
//   PV(1) S(3) | ..., so the tensor core computes PV(j) and S(j+2) while the
//   softmax works on S(j+1).
// The chunk's normalised O_s (float32) and LSE_s (log2 units) go to the
// workspace; fa_decode_combine_kernel merges the chunks exactly.
// Roles (256 threads): warp 0 TMA (Q once; K / V tiles in consumption order
// through a ring), warp 1 TMEM allocation and the MMA issuer, warps 4-7 the
// softmax (one query row per thread), then the chunk's epilogue.
// d = 256: O takes 256 TMEM columns (S_a 128 | S_b 128 | O 256), a K or V
// tile 64 KB, so K and V move through the ring in 128-feature halves (five
// 32 KB slots beside the 64 KB Q tile); S(j) runs over both halves of K_j
// (16 K-steps) and PV(j) is two N = 128 products, one per half of V_j and O.
// Causal (queries are the last Nq of Nk positions): key j is visible to
// query i iff j <= i + Nk - Nq; tiles past the query tile's last visible key
// are not read, a chunk no query of the tile sees writes LSE_s = -inf.
// Grouped queries (several query heads per K / V head): the query heads of
// one K / V head are consecutive in memory, so their rows form one longer
// query block of that head; row R of it is query R % qph (qph queries per
// head) of query head R / qph, and only the causal position uses qph.
#include "fa_decode.h"
#include "fa_fwd_kernel.cuh"

namespace fa {
namespace {

template <int D>
struct DecTcCfg {
  static constexpr int BM = 128;                   // queries per CTA (MMA M)
  static constexpr int BN = 128;                   // keys per tile
  static constexpr int SLABS = D / 64;
  static constexpr int SLAB = 128 * 128;           // 128 rows x 64 columns x 16 bit
  static constexpr int TILE = SLABS * SLAB;        // the Q tile
  static constexpr bool HALVES = D == 256;         // K / V in 128-feature halves
  static constexpr int PER = HALVES ? 2 : 1;       // ring items per K or V tile
  static constexpr int ITEM_SLABS = SLABS / PER;
  static constexpr int ITEM = ITEM_SLABS * SLAB;   // one ring slot
  static constexpr int NS = D == 256 ? 5 : (D == 128 ? 4 : 8);  // ring slots
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = TILE;
  static constexpr int OFF_BAR = OFF_RING + NS * ITEM;
  // q_full, ring_full[NS], ring_empty[NS], s_full[2], p_full[2], pv_done[2], o_full, drain
  static constexpr int NBAR = 1 + 2 * NS + 6 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;    // S_a at 0, S_b at 128
  static constexpr uint32_t COL_O = 256;  // D columns
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Ring position p of the consumption order K0, K1, V0, K2, V1, K3, ... for n
// tiles -> (is V, tile).
__device__ __forceinline__ void dec_ring_item(int p, int n, bool& is_v, int& tile) {
  const int first = n < 2 ? n : 2;  // K tiles before the first V
  if (p < first) {
    is_v = false;
    tile = p;
    return;
  }
  const int q = p - first;
  const int pairs = n - 2 > 0 ? n - 2 : 0;  // V_j followed by K_(j+2)
  if (q < 2 * pairs) {
    is_v = (q & 1) == 0;
    tile = is_v ? q / 2 : q / 2 + 2;
  } else {
    is_v = true;
    tile = pairs + (q - 2 * pairs);
  }
}

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(256, 1)
    fa_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, float* __restrict__ o_part,
                        float* __restrict__ lse_part, int Nq, int qph, int Nk, int BH, int chunk,
                        float scale_log2, unsigned int* status) {
  using C = DecTcCfg<D>;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int q0 = blockIdx.z * C::BM;        // rows of this K / V head: Nq = query heads x qph
  const int nq = min(C::BM, Nq - q0);
  const int off = Nk - qph;  // causal: key visible iff key <= position + off
  // query positions of the tile's rows (row R at position R % qph)
  const int p0 = q0 % qph;
  const bool wraps = p0 + nq > qph;  // the tile spans two query heads
  const int pmin = wraps ? 0 : p0;
  const int pmax = wraps ? qph - 1 : p0 + nq - 1;
  const int kb = split * chunk;
  int ke = min(Nk, kb + chunk);
  if (CAUSAL) ke = min(ke, pmax + 1 + off);  // one past the last key the tile's rows see
  const int n = ke > kb ? (ke - kb + C::BN - 1) / C::BN : 0;
  const long long part_row = (long long)split * BH * Nq + (long long)bh * Nq + q0;
  if (n == 0) {  // no query of this tile sees a key of the chunk: weight 0 in the combine
    for (int e = threadIdx.x; e < nq * D; e += blockDim.x) o_part[part_row * D + e] = 0.f;
    for (int e = threadIdx.x; e < nq; e += blockDim.x) lse_part[part_row + e] = neg_inf();
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sRing = smem + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* ring_full = q_full + 1;
  uint64_t* ring_empty = ring_full + C::NS;
  uint64_t* s_full = ring_empty + C::NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_full = pv_done + 2;
  uint64_t* drain = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
    }
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
  const int n_items = 2 * n * C::PER;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, C::TILE);
      for (int s = 0; s < C::SLABS; ++s) tma_load_3d(sQ + s * C::SLAB, &tm_q, q_full, s * 64, q0, bh);
      int issued = 0;
      for (int p = 0; p < n_items; ++p) {
        const int slot = p % C::NS;
        if (!mbar_wait(&ring_empty[slot], ((p / C::NS) & 1) ^ 1, abort_flag, status, kStatusTimeout)) break;
        bool is_v;
        int t;
        dec_ring_item(p / C::PER, n, is_v, t);
        const int half = p % C::PER;
        mbar_arrive_expect_tx(&ring_full[slot], C::ITEM);
        for (int s = 0; s < C::ITEM_SLABS; ++s)
          tma_load_3d(sRing + slot * C::ITEM + s * C::SLAB, is_v ? &tm_v : &tm_k, &ring_full[slot],
                      (half * C::ITEM_SLABS + s) * 64, kb + t * C::BN, bh);
        issued = p + 1;
      }
      if (*abort_flag) {
        drain_wait(q_full, 0);
        for (int p = issued - C::NS < 0 ? 0 : issued - C::NS; p < issued; ++p)
          drain_wait(&ring_full[p % C::NS], (uint32_t)((p / C::NS) & 1));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, C::BN, BF16, false, false);
      constexpr uint32_t kIdPV = idesc_f16(128, D / C::PER, BF16, false, true);
      const uint32_t aq = smem_u32(sQ), ring = smem_u32(sRing);
      int p = 0;  // ring position of the next item
      auto take = [&](int& slot) {
        slot = p % C::NS;
        const bool ok = mbar_wait(&ring_full[slot], (p / C::NS) & 1, abort_flag, status, kStatusTimeout);
        ++p;
        return ok;
      };
      // takes the ring slots of the next K or V tile (PER items)
      auto take_tile = [&](int (&sl)[C::PER]) {
        for (int h = 0; h < C::PER; ++h)
          if (!take(sl[h])) return false;
        tc_fence_after();
        return true;
      };
      auto issue_s = [&](int b, const int (&sl)[C::PER]) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int h = kk / (D / 16 / C::PER);  // the K slot holding K-step kk
          const int kl = kk % (D / 16 / C::PER);
          const uint32_t oa = (kk >> 2) * C::SLAB + (kk & 3) * 32;
          const uint32_t ob = (kl >> 2) * C::SLAB + (kl & 3) * 32;
          mma_ss(tmem + C::COL_S + 128 * b, sdesc_sw128(aq + oa, 16, 1024),
                 sdesc_sw128(ring + sl[h] * C::ITEM + ob, 16, 1024), kIdS, kk > 0);
        }
        mma_commit(&s_full[b]);
        for (int h = 0; h < C::PER; ++h) mma_commit(&ring_empty[sl[h]]);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, status, kStatusTimeout);
      int sl[C::PER];
      if (ok && (ok = take_tile(sl))) issue_s(0, sl);
      if (ok && n > 1 && (ok = take_tile(sl))) issue_s(1, sl);
      for (int j = 0; ok && j < n; ++j) {
        const int b = j & 1;
        if (!(ok = mbar_wait(&p_full[b], (j >> 1) & 1, abort_flag, status, kStatusTimeout))) break;
        if (!(ok = take_tile(sl))) break;  // V_j
        for (int h = 0; h < C::PER; ++h) {  // O (or its feature half h) += P V_j
          const uint64_t dv = sdesc_sw128(ring + sl[h] * C::ITEM, C::SLAB, 1024);
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            mma_ts(tmem + C::COL_O + (D / C::PER) * h, tmem + C::COL_S + 128 * b + 8 * kk,
                   dv + ((kk * 2048) >> 4), kIdPV, j > 0 || kk > 0);
        }
        mma_commit(&pv_done[b]);
        for (int h = 0; h < C::PER; ++h) mma_commit(&ring_empty[sl[h]]);
        // S(j+2) overwrites P(j): after PV(j), from the same thread (in order)
        if (j + 2 < n) {
          if (!(ok = take_tile(sl))) break;  // K_(j+2)
          issue_s(b, sl);
        }
      }
      if (ok) {
        mma_commit(o_full);
      } else {
        mma_commit(drain);
        drain_wait(drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax, epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int q_off = (q0 + r) % qph + off;  // causal: this row's key visible iff key <= q_off
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    float m_ref = neg_inf(), l = 0.f, l_mma = 0.f;
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      const uint32_t tS = lane_base + C::COL_S + 128 * b;
      if (!(ok = warp_wait(&s_full[b], (j >> 1) & 1, abort_flag, status))) break;
      tc_fence_after();
      float s[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + 32 * cc, s[cc]);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(s[cc]);
      const int kbase = kb + j * C::BN;
      const bool need_mask = (kbase + C::BN > ke) || (CAUSAL && kbase + C::BN - 1 > pmin + off);
      if (need_mask) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = kbase + 32 * cc + i;
            if (key >= ke || (CAUSAL && key > q_off)) s[cc][i] = neg_inf();
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
      const uint64_t nm2 = f2_pack(neg_m, neg_m);
      uint64_t sum2 = f2_pack(0.f, 0.f), sumr2 = f2_pack(0.f, 0.f);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
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
        tmem_st16(tS + 16 * cc, pk);
      }
      if (__any_sync(0xffffffffu, rescale_o)) {  // rare: PV(j-1) may still accumulate into O
        if (!(ok = warp_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, status))) break;
        tc_fence_after();
        if (rescale_o) {
          const uint64_t corr2 = f2_pack(corr, corr);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            float ov[32];
            tmem_ld32(lane_base + C::COL_O + 32 * cc, ov);
            tmem_ld_wait(ov);
            uint32_t ou[32];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float a, c2;
              f2_unpack(f2_mul(f2_pack(ov[i], ov[i + 1]), corr2), a, c2);
              ou[i] = __float_as_uint(a);
              ou[i + 1] = __float_as_uint(c2);
            }
            tmem_st32(lane_base + C::COL_O + 32 * cc, ou);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
      float a, c2;
      f2_unpack(sum2, a, c2);
      l += a + c2;
      f2_unpack(sumr2, a, c2);
      l_mma += a + c2;
    }
    // the chunk's normalised output (float32) and LSE (log2 units); a query
    // that sees no key of the chunk gets O_s = 0 and LSE_s = -inf (weight 0)
    if (ok) ok = warp_wait(o_full, 0, abort_flag, status);
    if (ok) {
      tc_fence_after();
      const float inv_l = l_mma > 0.f ? 1.f / l_mma : 0.f;
      float4* dst = reinterpret_cast<float4*>(o_part + (part_row + r) * D);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        float ov[32];
        tmem_ld32(lane_base + C::COL_O + 32 * cc, ov);
        tmem_ld_wait(ov);
        if (r < nq) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            dst[8 * cc + u] = make_float4(ov[4 * u] * inv_l, ov[4 * u + 1] * inv_l, ov[4 * u + 2] * inv_l,
                                          ov[4 * u + 3] * inv_l);
        }
      }
      if (r < nq) lse_part[part_row + r] = l > 0.f ? m_ref + __log2f(l) : neg_inf();
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
cudaError_t launch_dec_tc_t(const DecodeArgs& a, int qph, cudaStream_t stream) {
  using C = DecTcCfg<D>;
  auto kern = fa_decode_tc_kernel<D, CAUSAL, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.BH, (a.Nq + C::BM - 1) / C::BM);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.o_part, a.lse_part, a.Nq, qph, a.Nk,
                                               a.BH, a.chunk, a.scale_log2, a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc_grouped(int d, bool bf16, const DecodeArgs& a, int q_per_head, cudaStream_t stream) {
  if (q_per_head < 1 || a.Nq % q_per_head != 0) return cudaErrorInvalidValue;
#define FA_DEC_CASE(DD, CC, BB) \
  if (d == DD && a.causal == CC && bf16 == BB) return launch_dec_tc_t<DD, CC, BB>(a, q_per_head, stream);
  FA_DEC_CASE(64, false, false)
  FA_DEC_CASE(64, false, true)
  FA_DEC_CASE(64, true, false)
  FA_DEC_CASE(64, true, true)
  FA_DEC_CASE(128, false, false)
  FA_DEC_CASE(128, false, true)
  FA_DEC_CASE(128, true, false)
  FA_DEC_CASE(128, true, true)
  FA_DEC_CASE(256, false, false)
  FA_DEC_CASE(256, false, true)
  FA_DEC_CASE(256, true, false)
  FA_DEC_CASE(256, true, true)
#undef FA_DEC_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_tc(int d, bool bf16, const DecodeArgs& a, cudaStream_t stream) {
  return launch_decode_tc_grouped(d, bf16, a, a.Nq, stream);
}

}  // namespace fa

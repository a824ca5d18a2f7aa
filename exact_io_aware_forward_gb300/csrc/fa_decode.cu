// Split-KV forward for few queries against many keys (decoding) on the CUDA
// cores, used at d = 256 (d <= 128 runs the tensor-core kernel of
// fa_decode_tc.cu, which shares this file's workspace layout and combine).
//
// The key range of every head is cut into `num_splits` contiguous chunks; a
// CTA evaluates exact attention of up to QG queries over one chunk with the
// online-softmax recurrence ("FlashAttention 为什么不需要存下注意力矩阵",
// jefxiong.cn, section 3.2) and writes the chunk's normalised output O_s and
// its log-sum-exp LSE_s.  A second kernel merges the chunks exactly:
//   LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
// With Nq <= 16 queries a key row is used by at most 16 dot products, so the
// work is bound by streaming K and V from HBM; it runs on the CUDA cores:
//   scores   thread t <-> key t of a 256-key tile: 16-byte loads of its K row,
//            dot products with the (pre-scaled) queries held in shared memory;
//   softmax  block-wide max / sum per query (warp shuffles + shared memory),
//            running max and sum per query kept in every thread's registers;
//   P V      thread <-> (group of 8 features -- 4 for 16 queries --, a part of
//            the tile's keys): coalesced V loads, probabilities broadcast
//            from shared memory.
// Dot products and accumulations use the packed f32x2 FMA.
// Causal (queries are the last Nq of Nk positions): key j is visible to
// query i iff j <= i + Nk - Nq; chunks beyond a query group's last visible
// key are not read at all.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kTK = 256;       // keys per tile == threads per CTA
constexpr int kWarps = kTK / 32;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }

template <bool BF16>
__device__ __forceinline__ float2 to_f2(uint32_t w) {
  if (BF16) return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
  return __half22float2(*reinterpret_cast<__half2*>(&w));
}

template <bool BF16>
__device__ __forceinline__ uint32_t from_f2(float lo, float hi) {
  if (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Features per thread in the P V pass: 8 (one 16-byte V load per key) for up
// to 4 queries, 4 for 16 queries (register budget).
template <int QG>
struct DecodeFpt {
  static constexpr int value = QG <= 4 ? 8 : 4;
};

template <int D, int QG>
struct DecodeSmem {
  float q[QG][D];              // queries, pre-scaled by scale * log2(e)
  float p[QG][kTK];            // scores, then probabilities, of the current tile
  float red[kWarps][QG];       // per-warp partial max / sum
  float acc[kTK / (D / DecodeFpt<QG>::value)][QG][D];  // per key-part output partials
};

// One CTA: queries [q0, q0 + nq) of head bh against keys [kb, ke).
template <int D, bool BF16, bool CAUSAL, int QG>
__global__ void __launch_bounds__(kTK) fa_decode_split_kernel(
    const uint32_t* __restrict__ q, const uint4* __restrict__ k, const uint32_t* __restrict__ v,
    float* __restrict__ o_part, float* __restrict__ lse_part, int Nq, int Nk, int BH, int chunk,
    float scale_log2) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  auto& sm = *reinterpret_cast<DecodeSmem<D, QG>*>(smem_raw);
  constexpr int FPT = DecodeFpt<QG>::value;
  constexpr int NP = kTK / (D / FPT);  // key parts in the P V pass
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int q0 = blockIdx.z * QG;
  const int nq = min(QG, Nq - q0);
  const int kb = split * chunk;
  int ke = min(Nk, kb + chunk);
  if (CAUSAL) ke = min(ke, q0 + nq + Nk - Nq);  // past the group's last visible key
  const long long head_q = (long long)bh * Nq;
  const long long head_k = (long long)bh * Nk;

  for (int i = t; i < QG * D / 2; i += kTK) {
    const int qi = (2 * i) / D, f = (2 * i) % D;
    float2 x = make_float2(0.f, 0.f);
    if (qi < nq) x = to_f2<BF16>(q[((head_q + q0 + qi) * D + f) / 2]);
    sm.q[qi][f] = x.x * scale_log2;
    sm.q[qi][f + 1] = x.y * scale_log2;
  }
  float m[QG], l[QG];
  uint64_t acc[QG][FPT / 2];  // packed fp32 pairs of output features
#pragma unroll
  for (int i = 0; i < QG; ++i) {
    m[i] = neg_inf();
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < FPT / 2; ++e) acc[i][e] = f2_pack(0.f, 0.f);
  }
  const int fg = t % (D / FPT);  // feature group of the P V pass (FPT features)
  const int kp = t / (D / FPT);  // key part of the P V pass
  __syncthreads();

  for (int tile = kb; tile < ke; tile += kTK) {
    // ---- scores: thread t <-> key tile + t
    const int j = tile + t;
    float s[QG];
#pragma unroll
    for (int i = 0; i < QG; ++i) s[i] = 0.f;
    if (j < ke) {
      const uint4* krow = k + (head_k + j) * (D / 8);
      uint64_t s2[QG];  // packed partial dot products over even / odd features
#pragma unroll
      for (int i = 0; i < QG; ++i) s2[i] = f2_pack(0.f, 0.f);
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {
        const uint4 u = krow[c];
        const float2 k0 = to_f2<BF16>(u.x), k1 = to_f2<BF16>(u.y), k2 = to_f2<BF16>(u.z), k3 = to_f2<BF16>(u.w);
        const uint64_t kk0 = f2_pack(k0.x, k0.y), kk1 = f2_pack(k1.x, k1.y);
        const uint64_t kk2 = f2_pack(k2.x, k2.y), kk3 = f2_pack(k3.x, k3.y);
#pragma unroll
        for (int i = 0; i < QG; ++i) {
          const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&sm.q[i][8 * c]);
          const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(&sm.q[i][8 * c + 4]);
          s2[i] = f2_fma(kk0, a.x, f2_fma(kk1, a.y, f2_fma(kk2, b.x, f2_fma(kk3, b.y, s2[i]))));
        }
      }
#pragma unroll
      for (int i = 0; i < QG; ++i) {
        float lo, hi;
        f2_unpack(s2[i], lo, hi);
        s[i] = lo + hi;
      }
    }
#pragma unroll
    for (int i = 0; i < QG; ++i) {
      const bool vis = j < ke && i < nq && (!CAUSAL || j <= q0 + i + Nk - Nq);
      s[i] = vis ? s[i] : neg_inf();
    }
    // ---- tile max per query (block-wide)
#pragma unroll
    for (int i = 0; i < QG; ++i) {
      float x = s[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
      if (lane == 0) sm.red[warp][i] = x;
    }
    __syncthreads();
    float corr[QG];
#pragma unroll
    for (int i = 0; i < QG; ++i) {
      float x = sm.red[0][i];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) x = fmaxf(x, sm.red[w][i]);
      const float m_new = fmaxf(m[i], x);
      const float ref = m_new == neg_inf() ? 0.f : m_new;  // nothing visible yet
      corr[i] = m[i] == neg_inf() ? 0.f : exp2f(m[i] - ref);
      m[i] = m_new;
      s[i] = exp2f(s[i] - ref);  // exp2(-inf) = 0 for masked keys
      sm.p[i][t] = s[i];
    }
    __syncthreads();  // every thread has read sm.red; sm.p is complete
    // ---- tile sum per query (block-wide)
#pragma unroll
    for (int i = 0; i < QG; ++i) {
      float x = s[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      if (lane == 0) sm.red[warp][i] = x;
    }
    // ---- P V: thread <-> (feature group fg, keys kp, kp + NP, ...) of the tile
#pragma unroll
    for (int i = 0; i < QG; ++i) {
      const uint64_t c2 = f2_pack(corr[i], corr[i]);
#pragma unroll
      for (int e = 0; e < FPT / 2; ++e) acc[i][e] = f2_mul(acc[i][e], c2);
    }
    const int nk = min(kTK, ke - tile);
    const uint32_t* vrow0 = v + ((head_k + tile) * D) / 2 + fg * (FPT / 2);
#pragma unroll 4
    for (int jj = kp; jj < nk; jj += NP) {
      const uint32_t* vr = vrow0 + (long long)jj * (D / 2);
      uint64_t x[FPT / 2];
      if (FPT == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(vr);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < FPT / 2; ++e) {
          const float2 f = to_f2<BF16>(w[e]);
          x[e] = f2_pack(f.x, f.y);
        }
      } else {
        const uint2 u = *reinterpret_cast<const uint2*>(vr);
        const float2 f0 = to_f2<BF16>(u.x), f1 = to_f2<BF16>(u.y);
        x[0] = f2_pack(f0.x, f0.y);
        x[1] = f2_pack(f1.x, f1.y);
      }
#pragma unroll
      for (int i = 0; i < QG; ++i) {
        const float pij = sm.p[i][jj];
        const uint64_t p2 = f2_pack(pij, pij);
#pragma unroll
        for (int e = 0; e < FPT / 2; ++e) acc[i][e] = f2_fma(p2, x[e], acc[i][e]);
      }
    }
    __syncthreads();  // sm.red sums complete; sm.p no longer read
#pragma unroll
    for (int i = 0; i < QG; ++i) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) x += sm.red[w][i];
      l[i] = l[i] * corr[i] + x;
    }
    __syncthreads();  // sm.red free for the next tile
  }

  // ---- combine the key parts, normalise, write this chunk's O_s and LSE_s
#pragma unroll
  for (int i = 0; i < QG; ++i)
#pragma unroll
    for (int e = 0; e < FPT / 2; ++e) {
      float lo, hi;
      f2_unpack(acc[i][e], lo, hi);
      sm.acc[kp][i][fg * FPT + 2 * e] = lo;
      sm.acc[kp][i][fg * FPT + 2 * e + 1] = hi;
    }
  __syncthreads();
  const long long part_row = (long long)split * BH * Nq + head_q + q0;
  for (int e = t; e < QG * D; e += kTK) {
    const int i = e / D, f = e % D;
    if (i >= nq) continue;
    float x = 0.f;
#pragma unroll
    for (int pidx = 0; pidx < NP; ++pidx) x += sm.acc[pidx][i][f];
    o_part[(part_row + i) * D + f] = l[i] > 0.f ? x / l[i] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < QG; ++i)  // (static indices keep m and l in registers)
    if (t == i && i < nq) lse_part[part_row + i] = l[i] > 0.f ? m[i] + __log2f(l[i]) : neg_inf();
}

// One CTA per (head, query): LSE-weighted merge of the chunks (log2 domain in,
// natural log out).
template <int D, bool BF16>
__global__ void __launch_bounds__(D / 2) fa_decode_combine_kernel(const float* __restrict__ o_part,
                                                                 const float* __restrict__ lse_part,
                                                                 uint32_t* __restrict__ o, float* __restrict__ lse,
                                                                 int rows, int num_splits) {
  constexpr float kLn2 = 0.6931471805599453f;
  const long long row = blockIdx.x;  // bh * Nq + query
  const int f = 2 * threadIdx.x;
  float mx = neg_inf();
  for (int s = 0; s < num_splits; ++s) mx = fmaxf(mx, lse_part[(long long)s * rows + row]);
  const float ref = mx == neg_inf() ? 0.f : mx;
  float wsum = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll 8
  for (int s = 0; s < num_splits; ++s) {
    const float w = exp2f(lse_part[(long long)s * rows + row] - ref);  // 0 for chunks with nothing visible
    const float2 x = *reinterpret_cast<const float2*>(o_part + ((long long)s * rows + row) * D + f);
    wsum += w;
    a0 = fmaf(w, x.x, a0);
    a1 = fmaf(w, x.y, a1);
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  o[(row * D + f) / 2] = from_f2<BF16>(a0 * inv, a1 * inv);
  if (threadIdx.x == 0) lse[row] = (ref + __log2f(wsum)) * kLn2;
}

template <int D, bool BF16, bool CAUSAL, int QG>
cudaError_t launch_split_t(const DecodeArgs& a, cudaStream_t stream) {
  auto kern = fa_decode_split_kernel<D, BF16, CAUSAL, QG>;
  const int smem = (int)sizeof(DecodeSmem<D, QG>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.BH, (a.Nq + QG - 1) / QG);
  kern<<<grid, kTK, smem, stream>>>(static_cast<const uint32_t*>(a.q), static_cast<const uint4*>(a.k),
                                    static_cast<const uint32_t*>(a.v), a.o_part, a.lse_part, a.Nq, a.Nk, a.BH,
                                    a.chunk, a.scale_log2);
  return cudaGetLastError();
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_split_q(const DecodeArgs& a, cudaStream_t stream) {
  if (a.Nq == 1) return launch_split_t<D, BF16, CAUSAL, 1>(a, stream);
  if (a.Nq <= 4) return launch_split_t<D, BF16, CAUSAL, 4>(a, stream);
  return launch_split_t<D, BF16, CAUSAL, 16>(a, stream);
}

template <int D, bool BF16>
cudaError_t launch_combine_t(const DecodeArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.BH * a.Nq;
  if (rows > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_decode_combine_kernel<D, BF16><<<(unsigned)rows, D / 2, 0, stream>>>(
      a.o_part, a.lse_part, static_cast<uint32_t*>(a.o), a.lse, (int)rows, a.num_splits);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
  cudaError_t e = a.causal ? launch_split_q<D, BF16, true>(a, stream) : launch_split_q<D, BF16, false>(a, stream);
  if (e != cudaSuccess) return e;
  return launch_combine_t<D, BF16>(a, stream);
}

}  // namespace

int decode_default_splits(int BH, int Nq, int Nk) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long groups = (long long)BH * ((Nq + 15) / 16);
  const long long want = (16LL * sms + groups - 1) / groups;  // about sixteen CTAs per SM
  const long long max_splits = (Nk + 4 * kTK - 1) / (4 * kTK);  // at least four tiles per chunk
  long long s = want < max_splits ? want : max_splits;
  if (s > 1024) s = 1024;
  return s < 1 ? 1 : (int)s;
}

int decode_tc_default_splits(int BH, int Nq, int Nk) {
  // one CTA per SM (shared memory): about four waves of CTAs, at least eight
  // 128-key tiles per chunk
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long tiles = (long long)BH * ((Nq + 127) / 128);
  const long long want = (4LL * sms + tiles - 1) / tiles;
  const long long max_splits = (Nk + 1023) / 1024;
  long long s = want < max_splits ? want : max_splits;
  if (s > 1024) s = 1024;
  return s < 1 ? 1 : (int)s;
}

int decode_chunk(int Nk, int num_splits) {
  const int per = (Nk + num_splits - 1) / num_splits;
  return ((per + kTK - 1) / kTK) * kTK;
}

cudaError_t launch_decode_combine(int d, bool bf16, const DecodeArgs& a, cudaStream_t stream) {
  if (d == 64) return bf16 ? launch_combine_t<64, true>(a, stream) : launch_combine_t<64, false>(a, stream);
  if (d == 128) return bf16 ? launch_combine_t<128, true>(a, stream) : launch_combine_t<128, false>(a, stream);
  if (d == 256) return bf16 ? launch_combine_t<256, true>(a, stream) : launch_combine_t<256, false>(a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(int d, bool bf16, const DecodeArgs& a, cudaStream_t stream) {
  if (d == 64) return bf16 ? launch_decode_t<64, true>(a, stream) : launch_decode_t<64, false>(a, stream);
  if (d == 128) return bf16 ? launch_decode_t<128, true>(a, stream) : launch_decode_t<128, false>(a, stream);
  if (d == 256) return bf16 ? launch_decode_t<256, true>(a, stream) : launch_decode_t<256, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa

// Split-KV decoding (few queries against many keys): the chunk plan and the
// exact merge of the chunks.  The key range of every head is cut into
// `num_splits` contiguous chunks; the tensor-core kernel of fa_decode_tc.cu
// evaluates exact attention of a query tile over one chunk with the
// online-softmax recurrence ("FlashAttention 为什么不需要存下注意力矩阵",
// jefxiong.cn, section 3.2) and writes the chunk's normalised output O_s and
// its log-sum-exp LSE_s (log2 units) to the caller's workspace; the kernel
// here merges the chunks exactly:
//   LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kChunkKeys = 256;  // chunks are whole multiples of this many keys

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }

template <bool BF16>
__device__ __forceinline__ uint32_t from_f2(float lo, float hi) {
  if (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

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

template <int D, bool BF16>
cudaError_t launch_combine_t(const DecodeArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.BH * a.Nq;
  if (rows > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fa_decode_combine_kernel<D, BF16><<<(unsigned)rows, D / 2, 0, stream>>>(
      a.o_part, a.lse_part, static_cast<uint32_t*>(a.o), a.lse, (int)rows, a.num_splits);
  return cudaGetLastError();
}

}  // namespace

int decode_default_splits(int BH, int Nq, int Nk) {
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
  return ((per + kChunkKeys - 1) / kChunkKeys) * kChunkKeys;
}

cudaError_t launch_decode_combine(int d, bool bf16, const DecodeArgs& a, cudaStream_t stream) {
  if (d == 64) return bf16 ? launch_combine_t<64, true>(a, stream) : launch_combine_t<64, false>(a, stream);
  if (d == 128) return bf16 ? launch_combine_t<128, true>(a, stream) : launch_combine_t<128, false>(a, stream);
  if (d == 256) return bf16 ? launch_combine_t<256, true>(a, stream) : launch_combine_t<256, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa

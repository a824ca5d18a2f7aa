// Memory-bound helper kernels of the backward pass.
//
//   preprocess:  D_i = sum_c dO_ic * O_ic (float32) and, when an accumulator
//                is given, dq_accum := 0.
//                D replaces rowsum(P * (dO V^T)) of the softmax backward
//                ("FlashAttention 为什么不需要存下注意力矩阵", jefxiong.cn,
//                section 3.3): sum_j P_ij (dO_i . V_j) = dO_i . (P V)_i = dO_i . O_i.
//   dq_convert:  dQ = scale * dq_accum, rounded to the 16-bit type.
//
// Both stream over [rows, d] with 16-byte vector accesses; grids are a
// multiple of the SM count with grid-stride loops.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (BF16) {
      __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      float2 x = __bfloat1622float2(h);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 x = __half22float2(h);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// One row is handled by TPR consecutive threads (a power of two), VPT
// 16-byte vectors (8 elements) each: D = 64: 8 x 1, 96: 4 x 3, 128: 16 x 1,
// 256: 16 x 2.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const uint4* __restrict__ o,
                                                                const uint4* __restrict__ dO,
                                                                float* __restrict__ delta,
                                                                float4* __restrict__ dq_accum, long long rows) {
  constexpr int TPR = D == 96 ? 4 : D == 256 ? 16 : D / 8;
  constexpr int VPT = D / 8 / TPR;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int part = threadIdx.x % TPR;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  // The whole warp iterates together so that the row reduction can shuffle
  // across the full warp; lanes past the last row only idle.
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
       (t - (threadIdx.x & 31)) / TPR < rows; t += stride) {
    const long long row = t / TPR;
    const bool active = row < rows;
    const long long idx0 = active ? row * (D / 8) + part * VPT : 0;  // first 16-byte vector
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < VPT; ++u) {
      float a[8], b[8];
      unpack8<BF16>(o[idx0 + u], a);
      unpack8<BF16>(dO[idx0 + u], b);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(a[i], b[i], acc);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
    if (active) {
      if (part == 0) delta[row] = acc;
      if (dq_accum == nullptr) continue;  // D only (the split backward keeps no accumulator)
#pragma unroll
      for (int u = 0; u < VPT; ++u) {
        dq_accum[2 * (idx0 + u)] = zero;
        dq_accum[2 * (idx0 + u) + 1] = zero;
      }
    }
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float4* __restrict__ acc,
                                                                uint4* __restrict__ dq, long long n8,
                                                                float scale) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 x = acc[2 * i];
    const float4 y = acc[2 * i + 1];
    uint4 out;
    out.x = pack2<BF16>(x.x * scale, x.y * scale);
    out.y = pack2<BF16>(x.z * scale, x.w * scale);
    out.z = pack2<BF16>(y.x * scale, y.y * scale);
    out.w = pack2<BF16>(y.z * scale, y.w * scale);
    dq[i] = out;
  }
}

// The bounded pipeline wait of every kernel, on a barrier that never completes.
__global__ void fa_selftest_wait_kernel(unsigned int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  mbar_wait(&bar, 0, &abort_flag, status, kStatusTimeout);  // gives up after kWaitTimeoutNs
}

int grid_for(long long threads_needed) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long blocks = (threads_needed + 255) / 256;
  const long long cap = (long long)sms * 8;  // 8 resident 256-thread blocks per SM
  if (blocks <= 0) return 1;
  return (int)(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_backward_preprocess(int d, bool bf16, const void* o, const void* dO, float* delta,
                                       float* dq_accum, long long rows, cudaStream_t stream) {
  const long long threads = rows * (d == 96 ? 4 : d == 256 ? 16 : d / 8);
  const int grid = grid_for(threads);
  const uint4* o4 = static_cast<const uint4*>(o);
  const uint4* d4 = static_cast<const uint4*>(dO);
  float4* acc = reinterpret_cast<float4*>(dq_accum);
  if (d == 64 && bf16) fa_bwd_preprocess_kernel<64, true><<<grid, 256, 0, stream>>>(o4, d4, delta, acc, rows);
  else if (d == 64) fa_bwd_preprocess_kernel<64, false><<<grid, 256, 0, stream>>>(o4, d4, delta, acc, rows);
  else if (d == 96 && bf16) fa_bwd_preprocess_kernel<96, true><<<grid, 256, 0, stream>>>(o4, d4, delta, acc, rows);
  else if (d == 96) fa_bwd_preprocess_kernel<96, false><<<grid, 256, 0, stream>>>(o4, d4, delta, acc, rows);
  else if (d == 128 && bf16) fa_bwd_preprocess_kernel<128, true><<<grid, 256, 0, stream>>>(o4, d4, delta, acc, rows);
  else if (d == 128) fa_bwd_preprocess_kernel<128, false><<<grid, 256, 0, stream>>>(o4, d4, delta, acc, rows);
  else if (d == 256 && bf16) fa_bwd_preprocess_kernel<256, true><<<grid, 256, 0, stream>>>(o4, d4, delta, acc, rows);
  else if (d == 256) fa_bwd_preprocess_kernel<256, false><<<grid, 256, 0, stream>>>(o4, d4, delta, acc, rows);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait_timeout(unsigned int* status, cudaStream_t stream) {
  fa_selftest_wait_kernel<<<1, 1, 0, stream>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_backward_dq_convert(int d, bool bf16, const float* dq_accum, void* dq, long long rows,
                                       float scale, cudaStream_t stream) {
  const long long n8 = rows * d / 8;
  const int grid = grid_for(n8);
  const float4* acc = reinterpret_cast<const float4*>(dq_accum);
  uint4* out = static_cast<uint4*>(dq);
  if (bf16) fa_bwd_dq_convert_kernel<true><<<grid, 256, 0, stream>>>(acc, out, n8, scale);
  else fa_bwd_dq_convert_kernel<false><<<grid, 256, 0, stream>>>(acc, out, n8, scale);
  return cudaGetLastError();
}

}  // namespace fa

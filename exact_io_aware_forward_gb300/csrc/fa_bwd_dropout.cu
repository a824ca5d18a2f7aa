// dK / dV kernel with dropout: launch dispatch for the DROP instances of the
// kernel in fa_bwd_kernel.cuh, and the kernel that writes the keep mask
// itself (for callers and tests that want to see the mask).
#include "fa_bwd_kernel.cuh"

namespace fa {
namespace {

// One thread per 16 keys of one query row: one generator call.
__global__ void fa_dropout_keep_mask_kernel(uint8_t* __restrict__ keep, int BH, int Nq, int Nk, DropParams drop) {
  const int groups = (Nk + 15) / 16;
  const long long total = (long long)BH * Nq * groups;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(idx % groups);
    const long long rowid = idx / groups;  // bh * Nq + i
    const int i = (int)(rowid % Nq);
    const int bh = (int)(rowid / Nq);
    const uint4 w = philox4x32_10(make_uint4((uint32_t)g, (uint32_t)i, (uint32_t)bh, drop.offset), drop.k0, drop.k1);
    const uint32_t bits = keep_bits16(w, drop.t * 0x01010101u);
    uint8_t* dst = keep + rowid * Nk + 16LL * g;
    for (int k = 0; k < 16 && 16 * g + k < Nk; ++k) dst[k] = (uint8_t)((bits >> k) & 1u);
  }
}

}  // namespace

cudaError_t launch_backward_dkdv_dropout(int d, bool causal, bool bf16, const BwdArgs& a, cudaStream_t stream) {
#define FA_BWD_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_dkdv_t<DD, CC, BB, false, true, false>(a, stream);
  FA_BWD_CASE(64, false, false)
  FA_BWD_CASE(64, false, true)
  FA_BWD_CASE(64, true, false)
  FA_BWD_CASE(64, true, true)
  FA_BWD_CASE(128, false, false)
  FA_BWD_CASE(128, false, true)
  FA_BWD_CASE(128, true, false)
  FA_BWD_CASE(128, true, true)
  FA_BWD_CASE(256, false, false)
  FA_BWD_CASE(256, false, true)
  FA_BWD_CASE(256, true, false)
  FA_BWD_CASE(256, true, true)
#undef FA_BWD_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_dropout_keep_mask(uint8_t* keep, int BH, int Nq, int Nk, const DropParams& drop,
                                     cudaStream_t stream) {
  const long long total = (long long)BH * Nq * ((Nk + 15) / 16);
  if (total <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (total + 255) / 256;
  const int grid = (int)(want < 8LL * sms ? want : 8LL * sms);
  fa_dropout_keep_mask_kernel<<<grid, 256, 0, stream>>>(keep, BH, Nq, Nk, drop);
  return cudaGetLastError();
}

}  // namespace fa

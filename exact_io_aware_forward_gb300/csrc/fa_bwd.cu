// dK / dV kernel: launch dispatch for the dense and block-sparse instances of
// the kernel in fa_bwd_kernel.cuh.
#include "fa_bwd_kernel.cuh"

namespace fa {

int backward_q_tile(int d) { return d == 64 ? 128 : 64; }

namespace {

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_dkdv_s(const BwdArgs& a, cudaStream_t stream) {
  return a.block_mask ? launch_dkdv_t<D, CAUSAL, BF16, true, false, false>(a, stream)
                      : launch_dkdv_t<D, CAUSAL, BF16, false, false, false>(a, stream);
}

}  // namespace

cudaError_t launch_backward_dkdv(int d, bool causal, bool bf16, const BwdArgs& a, cudaStream_t stream) {
#define FA_BWD_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_dkdv_s<DD, CC, BB>(a, stream);
  FA_BWD_CASE(64, false, false)
  FA_BWD_CASE(64, false, true)
  FA_BWD_CASE(64, true, false)
  FA_BWD_CASE(64, true, true)
  FA_BWD_CASE(128, false, false)
  FA_BWD_CASE(128, false, true)
  FA_BWD_CASE(128, true, false)
  FA_BWD_CASE(128, true, true)
#undef FA_BWD_CASE
  // d = 256: dense only (no block-mask instance)
  if (d == 256 && !a.block_mask) {
    if (causal && bf16) return launch_dkdv_t<256, true, true, false, false, false>(a, stream);
    if (causal) return launch_dkdv_t<256, true, false, false, false, false>(a, stream);
    if (bf16) return launch_dkdv_t<256, false, true, false, false, false>(a, stream);
    return launch_dkdv_t<256, false, false, false, false, false>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa

// Forward pass: launch dispatch for dense layouts without dropout.  Block
// masks run the kernel in fa_fwd_kernel.cuh; plain dense attention runs the
// kernel of fa_fwd_persist.cu (Q with a producer of its own, per-query-tile
// O hand-off, persistent CTAs at d = 64).
#include "fa_fwd_kernel.cuh"

namespace fa {
namespace {

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_fwd_s(const FwdArgs& a, cudaStream_t stream) {
  return a.block_mask ? launch_fwd_t<D, CAUSAL, BF16, true, false, false>(a, stream)
                      : launch_forward_persistent(D, CAUSAL, BF16, a, stream);
}

}  // namespace

cudaError_t launch_forward(int d, bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream) {
#define FA_FWD_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_fwd_s<DD, CC, BB>(a, stream);
  FA_FWD_CASE(64, false, false)
  FA_FWD_CASE(64, false, true)
  FA_FWD_CASE(64, true, false)
  FA_FWD_CASE(64, true, true)
  FA_FWD_CASE(128, false, false)
  FA_FWD_CASE(128, false, true)
  FA_FWD_CASE(128, true, false)
  FA_FWD_CASE(128, true, true)
#undef FA_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa

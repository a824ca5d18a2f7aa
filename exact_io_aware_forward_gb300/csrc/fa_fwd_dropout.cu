// Forward pass with dropout: launch dispatch for the DROP instances of the
// kernel in fa_fwd_kernel.cuh (dense attention, keep bits regenerated from
// the Philox seed and offset).
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_forward_dropout(int d, bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream) {
#define FA_FWD_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_fwd_t<DD, CC, BB, false, true, false>(a, stream);
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

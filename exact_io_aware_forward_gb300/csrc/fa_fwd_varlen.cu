// Forward pass over packed variable-length batches: launch dispatch for the
// VARLEN instances of the kernel in fa_fwd_kernel.cuh (with and without
// dropout).
#include "fa_fwd_kernel.cuh"

namespace fa {
namespace {

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_fwd_v(const FwdArgs& a, cudaStream_t stream) {
  return a.dropout ? launch_fwd_t<D, CAUSAL, BF16, false, true, true>(a, stream)
                   : launch_fwd_t<D, CAUSAL, BF16, false, false, true>(a, stream);
}

}  // namespace

cudaError_t launch_forward_varlen(int d, bool causal, bool bf16, const FwdArgs& a, cudaStream_t stream) {
#define FA_FWD_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_fwd_v<DD, CC, BB>(a, stream);
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

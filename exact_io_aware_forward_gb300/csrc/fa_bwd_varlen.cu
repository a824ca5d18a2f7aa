// dK / dV kernel over packed variable-length batches: launch dispatch for the
// VARLEN instances of the kernel in fa_bwd_kernel.cuh (with and without
// dropout).
#include "fa_bwd_kernel.cuh"

namespace fa {
namespace {

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_dkdv_v(const BwdArgs& a, cudaStream_t stream) {
  return a.dropout ? launch_dkdv_t<D, CAUSAL, BF16, false, true, true>(a, stream)
                   : launch_dkdv_t<D, CAUSAL, BF16, false, false, true>(a, stream);
}

}  // namespace

cudaError_t launch_backward_dkdv_varlen(int d, bool causal, bool bf16, const BwdArgs& a, cudaStream_t stream) {
#define FA_BWD_CASE(DD, CC, BB) \
  if (d == DD && causal == CC && bf16 == BB) return launch_dkdv_v<DD, CC, BB>(a, stream);
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

}  // namespace fa

// dK/dV kernel of the backward pass (placeholder until the tcgen05 version lands).
#include "fa_internal.h"

namespace fa {
int backward_q_tile(int d) { return d == 128 ? 64 : 128; }
cudaError_t launch_backward_dkdv(int, bool, bool, const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa

// Launch interface of grouped-query decoding (several query heads per K / V
// head).  Not part of the public interface.
#pragma once

#include "fa_internal.h"

namespace fa {

// a.BH counts K / V heads and a.Nq the query rows of one K / V head (its
// query heads x q_per_head, consecutive in memory); a.tm_q maps q as
// [a.BH, a.Nq, d].  Query row R of a head sits at position R % q_per_head.
cudaError_t launch_decode_tc_grouped(int d, bool bf16, const DecodeArgs& a, int q_per_head, cudaStream_t stream);

}  // namespace fa

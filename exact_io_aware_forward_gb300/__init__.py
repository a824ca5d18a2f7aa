"""Exact IO-aware softmax attention for GB300 (sm_103a).

The compute lives in ``libfa_gb300.so`` (hand-written tcgen05/TMA kernels,
C ABI in ``include/fa_gb300.h``); ``api`` is its thin Python binding.
Importing this package does not load the library; the first call does, and
fails loudly if it has not been built.
"""
from .api import (FAError, backward, fa_backward, fa_backward_dkdv, fa_backward_dq_convert,  # noqa: F401
                  fa_backward_dk_dv, fa_backward_dq, fa_backward_dk_dv_blocksparse,
                  fa_backward_dq_blocksparse,
                  fa_backward_noalloc, fa_decode_workspace_size, fa_forward_decode, forward_decode,
                  fa_decode_gqa_workspace_size, fa_forward_decode_gqa,
                  fa_forward_blocksparse, fa_backward_blocksparse, fa_backward_dkdv_blocksparse,
                  fa_forward_dropout, fa_backward_dropout, fa_backward_dkdv_dropout, fa_dropout_keep_mask,
                  fa_backward_dk_dv_dropout, fa_backward_dq_dropout,
                  fa_forward_varlen, fa_backward_varlen, fa_backward_varlen_workspace_size, forward_varlen,
                  backward_varlen, fa_backward_dkdv_varlen, fa_backward_dk_dv_varlen, fa_backward_dq_varlen,
                  fa_selftest_wait_timeout,
                  fa_backward_preprocess, fa_backward_workspace_size, fa_device_status, fa_forward,
                  fa_score_blocks, forward)

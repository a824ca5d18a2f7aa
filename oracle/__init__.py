"""Float64 CPU oracle for exact softmax attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA library (no kernels,
headers, helpers or constants); the only thing both sides share is the seeded
input generator in ``exact_io_aware_forward_gb300.synth``, which holds none of
the attention arithmetic.

Modules
-------
``attention``  the plain definition, with S and P materialised (forward and
               the explicit softmax backward).
``online``     an independent streaming (online-softmax) evaluation used only
               to pin ``attention`` against the recurrence the pages derive.
``dropout``    the Philox4x32-10 counter-based generator (written from its
               published definition) and the keep mask it defines.
``varlen``     packed variable-length sequences: each sequence an independent
               problem, bottom-right causal alignment when Nq != Nk.

Every function cites the page passage it follows.  Pages are named by title:

* P1 -- "FlashAttention V1 技术深度解析" (spark.aweffr.cn lecture summary)
* P3 -- "FlashAttention 为什么不需要存下注意力矩阵" (jefxiong.cn tutorial)

Parity pins (all under ``tests/test_oracle*.py``): the page's worked trace
(P3 section 04.1), the page's exactness bound (P3 section 04.2), the page's
rescale ablation (P3 section 09), the causal block count (P3 section 04.5),
closed forms (uniform scores, causal row 0, N = 1), an independent
log-sum-exp, torch's float64 CPU attention and autograd, central finite
differences, the backward invariants that follow from P3 section 3.3, and
for dropout the generator's published known-answer values, a per-entry
scalar evaluation of the counter mapping, binomial bounds on the keep
fraction, and torch float64 autograd with the keep mask as a constant.
No function is "parity unpinned".
"""
from . import attention, dropout, online, varlen  # noqa: F401

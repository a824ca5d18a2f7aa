"""Attention over packed variable-length sequences.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages treat one sequence at a time (P3 section 3: every row block of Q
meets every column block of K and V of the same sequence).  A batch of
sequences of different lengths is read as independent problems laid end to
end: sequence b owns query rows cu_q[b] .. cu_q[b+1]-1 and key rows
cu_k[b] .. cu_k[b+1]-1 of the packed tensors, and no query ever sees a key of
another sequence.  Within a sequence the rules of ``oracle.attention`` hold,
including the bottom-right causal alignment for Nq != Nk (query i of the
sequence sits at position i + Nk_b - Nq_b) and O = 0, LSE = -inf for a query
that sees no key.

Layout: token-major packed tensors, q [Tq, H, d], k and v [Tk, H, d];
O [Tq, H, d] and LSE [Tq, H].
"""
from __future__ import annotations

import numpy as np

from . import attention as A


def _ranges(cu):
    cu = np.asarray(cu, dtype=np.int64)
    return [(int(cu[b]), int(cu[b + 1])) for b in range(len(cu) - 1)]


def forward_varlen(q, k, v, cu_q, cu_k, scale, causal=False):
    """O [Tq, H, d] and LSE [Tq, H] of every sequence and head."""
    Tq, H, _ = q.shape
    o = np.zeros((Tq, H, v.shape[-1]))
    lse = np.full((Tq, H), -np.inf)
    for (q0, q1), (k0, k1) in zip(_ranges(cu_q), _ranges(cu_k)):
        if q1 == q0:
            continue
        for h in range(H):
            if k1 == k0:  # no key at all: every row is empty
                continue
            o[q0:q1, h], lse[q0:q1, h] = A.forward_head(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], scale, causal)
    return o, lse


def backward_varlen(q, k, v, do, cu_q, cu_k, scale, causal=False):
    """(dQ [Tq, H, d], dK [Tk, H, d], dV [Tk, H, d])."""
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    H = q.shape[1]
    for (q0, q1), (k0, k1) in zip(_ranges(cu_q), _ranges(cu_k)):
        if q1 == q0 or k1 == k0:
            continue
        for h in range(H):
            dq[q0:q1, h], dk[k0:k1, h], dv[k0:k1, h] = A.backward_head(
                q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], do[q0:q1, h], scale, causal)
    return dq, dk, dv

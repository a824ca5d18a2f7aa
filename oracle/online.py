"""Streaming (online-softmax) evaluation of one attention head, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  This exists to pin
``oracle.attention`` against the recurrence the pages derive; it is not a
model of the CUDA kernel and shares no code with ``oracle.attention``.

Recurrence (P3 "FlashAttention 为什么不需要存下注意力矩阵", section 3.2):
keys arrive in blocks; for every query row keep the reference max m, the
denominator l and the unnormalised accumulator O.  When block t+1 arrives
with block max m_blk:

    m' = max(m, m_blk)
    l' = exp(m - m') * l + sum_blk exp(s - m')
    O' = exp(m - m') * O + sum_blk exp(s - m') v

starting from m = -inf, l = 0, O = 0 with the factor exp(m - m') taken as 0
while m is still -inf.  The result is O / l and the LSE is m + log l.
Masked (causal) scores are -inf and contribute nothing (same section); with
fewer queries than keys the queries are the last positions.

Here all query rows advance together and keys stream in blocks of
``block`` rows (1 = one key at a time, the Milakov-Gimelshein online
normaliser the page cites in section 07).
"""
from __future__ import annotations

import numpy as np


def online_attention(q, k, v, block, scale=None, causal=False, trace_row=None,
                     rescale=True):
    """Return (O, LSE, trace) for one head [N, d].

    ``trace`` lists (first key of block, m, l, factor) for query
    ``trace_row`` after every block, as printed in P3 section 04.1.
    ``rescale=False`` replaces the factor exp(m - m') by 1: the ablation of
    P3 section 09, which must make the result wrong.
    """
    n_q, d = q.shape
    n_k = k.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    m = np.full(n_q, -np.inf)
    l = np.zeros(n_q)
    acc = np.zeros((n_q, v.shape[1]))
    trace = []
    query_idx = np.arange(n_q) + (n_k - n_q)  # query positions (last n_q of n_k)
    for j0 in range(0, n_k, block):
        j1 = min(n_k, j0 + block)
        s = scale * (q @ k[j0:j1].T)                      # [n_q, blk]
        if causal:
            key_idx = np.arange(j0, j1)
            s = np.where(key_idx[None, :] > query_idx[:, None], -np.inf, s)
        m_new = np.maximum(m, s.max(axis=1))
        if rescale:
            with np.errstate(invalid="ignore"):
                factor = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
        else:
            factor = np.ones(n_q)
        w = np.exp(s - m_new[:, None])                    # block weights
        l = factor * l + w.sum(axis=1)
        acc = factor[:, None] * acc + w @ v[j0:j1]
        m = m_new
        if trace_row is not None:
            trace.append((j0, float(m[trace_row]), float(l[trace_row]),
                          float(factor[trace_row])))
    return acc / l[:, None], m + np.log(l), trace


def causal_blocks_kept(N, B_r, B_c):
    """Blocks visited under the causal whole-block skip (P3 section 04.5).

    A (query block, key block) pair is skipped when every query index of the
    block is below every key index of the key block.
    """
    kept = 0
    for i0 in range(0, N, B_r):
        for j0 in range(0, N, B_c):
            q_last = min(N, i0 + B_r) - 1
            if q_last < j0:
                continue
            kept += 1
    return kept

"""Plain float64 softmax attention with S and P materialised.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Definitions followed
--------------------
* Forward: P1 section 2.1 (Attention = softmax(QK^T/sqrt(d_k)) V) and P3
  section 3.1 (safe softmax: subtract the row max, exponentiate, divide by
  the row sum).  The scale ``s`` is a parameter; the pages use 1/sqrt(d).
* Causal mask: P3 section 3.2 (masked scores are set to -inf so they add
  nothing to m, l or O); key j is visible to query i iff j <= i (square
  problem).  With Nq queries and Nk >= Nq keys (decoding) the queries are
  read as the last Nq positions: key j is visible to query i iff
  j <= i + Nk - Nq, which is the square rule when Nq = Nk.
* LSE: P3 section 3.2, natural log: LSE_i = m_i + log(l_i) with m_i the row
  max of the *scaled* scores.
* Backward: P3 section 3.3 -- with G = dO and A = G V^T,
  dS = P * (A - rowsum(A * P)), dQ = s * dS K, dK = s * dS^T Q, dV = P^T G.
  The row sum is taken over A * P exactly as written there, not through the
  rowsum(dO * O) shortcut the CUDA path uses.

* Block-sparse attention (P3 section 06: the whole-block skip generalised to
  any sparsity pattern): a boolean block mask over 128 x 128 (query, key)
  blocks removes whole blocks, i.e. their scores are -inf like masked causal
  scores.  A query row with no visible key at all has no softmax; the
  reading taken is O = 0 and LSE = -inf for it (and no gradient flows).

* Dropout (P3 section 05: the mask is regenerated from the generator's seed
  and offset, never stored): with a boolean keep mask Z and the keep scale
  c = 1 / keep probability, the forward pass uses P~ = P * Z * c in place of
  P, so O = P~ V, while LSE stays the softmax normaliser of the undropped
  scores.  Backward: dV = P~^T G; the gradient reaching P is
  dP = (G V^T) * Z * c, and dS = P * (dP - rowsum(dP * P)).  Z itself comes
  from ``oracle.dropout``.

Arrays are numpy float64.  Batched entry points take [B, H, N, d] arrays and
loop over heads; the ``*_head`` functions take one head [N, d].
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# building blocks (kept separate so that tests can plant mistakes in them)
# --------------------------------------------------------------------------
BLOCK = 128  # rows / columns of one block of a block mask


def _scores(q, k, scale, causal, rows=None, block_mask=None):
    """S = s * Q K^T for the query rows ``rows`` (all rows if None).

    Causal: entries with key index > query position become -inf (P3 section
    3.2); query i sits at position i + Nk - Nq.  ``block_mask`` (boolean,
    [ceil(Nq/128), ceil(Nk/128)]): entries of blocks marked False become -inf.
    """
    if rows is None:
        rows = np.arange(q.shape[0])
    rows = np.asarray(rows)
    s = scale * (q[rows] @ k.T)
    if causal:
        keys = np.arange(k.shape[0])
        pos = rows + (k.shape[0] - q.shape[0])
        s = np.where(keys[None, :] > pos[:, None], -np.inf, s)
    if block_mask is not None:
        bm = np.asarray(block_mask, dtype=bool)
        keep = bm[rows // BLOCK][:, np.arange(k.shape[0]) // BLOCK]
        s = np.where(keep, s, -np.inf)
    return s


def _softmax_rows(s):
    """Safe softmax of every row (P3 section 3.1).

    Returns (P, m, l) with m the row max and l = sum exp(s - m).  A row whose
    scores are all -inf (no visible key) gets P = 0, m = -inf, l = 0.
    """
    m = s.max(axis=1)
    empty = np.isneginf(m)
    e = np.exp(s - np.where(empty, 0.0, m)[:, None])
    l = e.sum(axis=1)
    return e / np.where(empty, 1.0, l)[:, None], m, l


def _softmax_backward(p, a):
    """dS = P * (A - rowsum(A * P)) (P3 section 3.3)."""
    return p * (a - (a * p).sum(axis=1, keepdims=True))


# --------------------------------------------------------------------------
# one head
# --------------------------------------------------------------------------
def _dropped(p, keep, keep_scale):
    """P~ = P * Z * c (P itself when there is no dropout)."""
    if keep is None:
        return p
    return np.where(keep, p * keep_scale, 0.0)


def forward_head(q, k, v, scale, causal=False, rows=None, block_mask=None, keep=None, keep_scale=1.0):
    """O and LSE of one head ([N, d] inputs) for the query rows ``rows``.

    ``keep`` (boolean [rows, Nk]) and ``keep_scale`` apply dropout to P."""
    s = _scores(q, k, scale, causal, rows, block_mask)
    p, m, l = _softmax_rows(s)
    with np.errstate(divide="ignore"):
        return _dropped(p, keep, keep_scale) @ v, m + np.log(l)


def probabilities_head(q, k, scale, causal=False, rows=None):
    """The full softmax matrix P of one head (for invariant checks)."""
    p, _, _ = _softmax_rows(_scores(q, k, scale, causal, rows))
    return p


def backward_head(q, k, v, do, scale, causal=False, block_mask=None, keep=None, keep_scale=1.0):
    """(dQ, dK, dV) of one head, everything materialised (P3 section 3.3).

    With dropout (``keep``, ``keep_scale``) the gradient reaching P is
    (dO V^T) * Z * c and dV = P~^T dO."""
    p, _, _ = _softmax_rows(_scores(q, k, scale, causal, block_mask=block_mask))
    a = _dropped(do @ v.T, keep, keep_scale)
    ds = _softmax_backward(p, a)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    dv = _dropped(p, keep, keep_scale).T @ do
    return dq, dk, dv


def backward_head_sampled(q, k, v, do, scale, causal, rows, cols, stripe=2048):
    """dQ at query rows ``rows`` and dK, dV at key rows ``cols`` of one head.

    The same definition as ``backward_head``; S, P and A are built in stripes
    of ``stripe`` query rows so that a long head fits in host memory.  dK and
    dV at a key j need column j of dS for every query, so every stripe is
    visited; dQ at a query i needs only row i.
    """
    n = q.shape[0]
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    dk = np.zeros((len(cols), q.shape[1]))
    dv = np.zeros((len(cols), v.shape[1]))
    for r0 in range(0, n, stripe):
        r = np.arange(r0, min(n, r0 + stripe))
        p, _, _ = _softmax_rows(_scores(q, k, scale, causal, r))
        a = do[r] @ v.T
        ds = _softmax_backward(p, a)
        dk += scale * (ds[:, cols].T @ q[r])
        dv += p[:, cols].T @ do[r]
    return backward_head_rows(q, k, v, do, scale, causal, rows), dk, dv


def backward_head_rows(q, k, v, do, scale, causal, rows):
    """dQ at query rows ``rows`` of one head: row i of dS needs only row i of
    S, P and A = dO V^T (Tutorial section 3.3), so this costs O(len(rows) N d)."""
    rows = np.asarray(rows)
    p, _, _ = _softmax_rows(_scores(q, k, scale, causal, rows))
    ds = _softmax_backward(p, do[rows] @ v.T)
    return scale * (ds @ k)


# --------------------------------------------------------------------------
# batched [B, H, N, d]
# --------------------------------------------------------------------------
def forward(q, k, v, scale, causal=False):
    """O [B,H,N,d] and LSE [B,H,N] of every head."""
    B, H, N, d = q.shape
    o = np.empty((B, H, N, v.shape[-1]))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal)
    return o, lse


def backward(q, k, v, do, scale, causal=False):
    """dQ, dK, dV [B,H,N,d] of every head."""
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = backward_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
    return dq, dk, dv

"""Pins of the packed variable-length oracle and of the rectangular
(Nq != Nk, bottom-right causal) backward (no GPU).

Independent formulation: the whole packed batch as ONE attention problem per
head under a block-diagonal mask (bottom-right causal inside each block),
evaluated by torch's float64 attention and autograd.
"""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import varlen as VL


def _packed_mask(cu_q, cu_k, causal):
    """Boolean [Tq, Tk]: query row r sees key column c."""
    Tq, Tk = cu_q[-1], cu_k[-1]
    m = np.zeros((Tq, Tk), bool)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        blk = np.ones((q1 - q0, k1 - k0), bool)
        if causal:
            blk = np.tril(blk, k=(k1 - k0) - (q1 - q0))
        m[q0:q1, k0:k1] = blk
    return m


def _torch_packed(q, k, v, do, mask, scale):
    """Per head: softmax over the masked packed scores; rows without any
    visible key are left out of the loss (torch gives NaN there)."""
    H = q.shape[1]
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))  # [H, T, d]
    tm = torch.tensor(mask)
    s = scale * tq @ tk.transpose(1, 2)
    s = s.masked_fill(~tm, float("-inf"))
    live = tm.any(dim=1)  # [Tq]
    p = torch.softmax(s[:, live], dim=-1)
    o = torch.zeros(H, q.shape[0], v.shape[2], dtype=torch.float64)
    o[:, live] = p @ tv
    lse = torch.full((H, q.shape[0]), float("-inf"), dtype=torch.float64)
    lse[:, live] = torch.logsumexp(s[:, live], dim=-1)
    o.backward(torch.tensor(do.transpose(1, 0, 2)))
    t = lambda x: x.detach().numpy().transpose(1, 0, 2)  # noqa: E731
    return t(o), lse.detach().numpy().T, t(tq.grad), t(tk.grad), t(tv.grad)


CASES = [  # (query lengths, key lengths)
    ([5, 17, 1, 30], [5, 17, 1, 30]),
    ([3, 40, 12], [20, 41, 12]),      # Nq <= Nk: decoding-like tails
    ([9, 2, 25], [4, 2, 30]),          # Nq > Nk in the first sequence: empty causal rows
    ([0, 7, 3], [5, 0, 9]),            # an empty query range and an empty key range
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lq,lk", CASES)
def test_varlen_against_packed_torch(causal, lq, lk):
    rng = np.random.default_rng(sum(lq) * 7 + sum(lk))
    H, d, s = 3, 8, 0.4
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int64)
    q = rng.normal(size=(cu_q[-1], H, d))
    k, v = rng.normal(size=(cu_k[-1], H, d)), rng.normal(size=(cu_k[-1], H, d))
    do = rng.normal(size=q.shape)
    o, lse = VL.forward_varlen(q, k, v, cu_q, cu_k, s, causal)
    dq, dk, dv = VL.backward_varlen(q, k, v, do, cu_q, cu_k, s, causal)
    to, tlse, tdq, tdk, tdv = _torch_packed(q, k, v, do, _packed_mask(cu_q, cu_k, causal), s)
    assert np.abs(o - to).max() < 1e-12
    assert np.array_equal(np.isneginf(lse), np.isneginf(tlse))
    fin = np.isfinite(tlse)
    assert np.abs(lse[fin] - tlse[fin]).max() < 1e-12
    for g, t in ((dq, tdq), (dk, tdk), (dv, tdv)):
        assert np.abs(g - t).max() < 1e-11


def test_single_sequence_equals_dense():
    rng = np.random.default_rng(3)
    N, H, d = 37, 2, 4
    q, k, v, do = (rng.normal(size=(N, H, d)) for _ in range(4))
    cu = np.array([0, N])
    for causal in (False, True):
        o, lse = VL.forward_varlen(q, k, v, cu, cu, 0.5, causal)
        dq, dk, dv = VL.backward_varlen(q, k, v, do, cu, cu, 0.5, causal)
        for h in range(H):
            ro, rl = A.forward_head(q[:, h], k[:, h], v[:, h], 0.5, causal)
            assert np.array_equal(o[:, h], ro) and np.array_equal(lse[:, h], rl)
            for g, r in zip((dq, dk, dv), A.backward_head(q[:, h], k[:, h], v[:, h], do[:, h], 0.5, causal)):
                assert np.array_equal(g[:, h], r)


@pytest.mark.parametrize("Nq,Nk", [(1, 9), (6, 40), (40, 6), (33, 33)])
def test_rectangular_backward_against_torch(Nq, Nk):
    """The bottom-right causal backward of one head equals torch autograd with
    the explicit mask (rows without a visible key left out)."""
    rng = np.random.default_rng(Nq + 100 * Nk)
    d, s = 8, 0.35
    q, do = rng.normal(size=(Nq, 1, d)), rng.normal(size=(Nq, 1, d))
    k, v = rng.normal(size=(Nk, 1, d)), rng.normal(size=(Nk, 1, d))
    mask = np.tril(np.ones((Nq, Nk), bool), k=Nk - Nq)
    to, tlse, tdq, tdk, tdv = _torch_packed(q, k, v, do, mask, s)
    o, lse = A.forward_head(q[:, 0], k[:, 0], v[:, 0], s, True)
    dq, dk, dv = A.backward_head(q[:, 0], k[:, 0], v[:, 0], do[:, 0], s, True)
    assert np.abs(o - to[:, 0]).max() < 1e-12
    for g, t in ((dq, tdq), (dk, tdk), (dv, tdv)):
        assert np.abs(g - t[:, 0]).max() < 1e-11


def test_planted_top_left_alignment_is_caught(monkeypatch):
    """A top-left causal rule for Nq != Nk (key j visible iff j <= i) fails the
    packed pin."""
    lq, lk = [3, 40, 12], [20, 41, 12]
    rng = np.random.default_rng(5)
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    q = rng.normal(size=(cu_q[-1], 2, 8))
    k, v = rng.normal(size=(cu_k[-1], 2, 8)), rng.normal(size=(cu_k[-1], 2, 8))
    real = A._scores

    def top_left(q_, k_, scale, causal, rows=None, block_mask=None):
        s = real(q_, k_, scale, False, rows, block_mask)
        if causal:
            r = np.arange(q_.shape[0]) if rows is None else np.asarray(rows)
            s = np.where(np.arange(k_.shape[0])[None, :] > r[:, None], -np.inf, s)
        return s

    monkeypatch.setattr(A, "_scores", top_left)
    o, _ = VL.forward_varlen(q, k, v, cu_q, cu_k, 0.4, True)
    to, *_ = _torch_packed(q, k, v, np.zeros_like(q), _packed_mask(cu_q, cu_k, True), 0.4)
    assert np.abs(o - to).max() > 1e-3

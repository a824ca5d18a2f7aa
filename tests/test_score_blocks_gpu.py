"""Work counters: the score tiles the kernels compute (whole-tile causal skip,
block-sparse skip) against closed forms.

"FlashAttention 为什么不需要存下注意力矩阵" (jefxiong.cn), section 04.5: a tile
that lies wholly above the causal diagonal is skipped, so T(T+1)/2 of the T x T
square tiles are visited (2080 of 4096 at 64-row blocks and N = 4096; at the
kernels' 128-row tiles the same rule gives 528 of 1024).  The counters count
64 x 64 score blocks, so a 128 x 128 tile is 4 of them.

The dense forward at d <= 128 runs query tiles in pairs: with an odd number
T of query tiles the second tile of the last pair starts past the last row
and still runs its T key tiles (its rows are never stored).  Skipping it in
the kernel measured slower on the even-T workloads, so the count includes it.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import attention_inputs, varlen_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _tri(T):
    return T * (T + 1) // 2


def _fwd_expected(T, causal, d):
    """Forward blocks of one head, N = 128 T (square)."""
    tiles = _tri(T) if causal else T * T
    phantom = T if (T % 2 == 1 and d != 256) else 0
    return 4 * (tiles + phantom)


def _counts(fn):
    fa.fa_score_blocks(reset=True)
    fn()
    fa.fa_device_status()
    return fa.fa_score_blocks(reset=True)


def _fwd_bwd_counts(B, H, N, d, causal, dtype="bf16", block_mask=None):
    q, k, v, do = (x.to(DEV) for x in attention_inputs(B, H, N, d, dtype, seed=N + d))
    md = None if block_mask is None else torch.from_numpy(block_mask.astype(np.uint8)).to(DEV)
    out = {}

    def fwd():
        out["o"], out["lse"] = fa.forward(q, k, v, causal=causal, block_mask=md)

    def bwd():
        fa.backward(q, k, v, out["o"], out["lse"], do, causal=causal, block_mask=md)

    f, b = _counts(fwd)
    assert b == 0
    f2, b2 = _counts(bwd)
    assert f2 == 0
    return f, b2


@pytest.mark.parametrize("d", [64, 96, 128, 256])
@pytest.mark.parametrize("T", [1, 3, 4, 7])
def test_causal_skip_visits_T_T_plus_1_over_2(d, T):
    """Square causal problems, N = 128 T: the backward computes 4 BH T(T+1)/2
    blocks, the forward the same plus the unpaired tile's at odd T."""
    B, H = 1, 3
    f, b = _fwd_bwd_counts(B, H, 128 * T, d, causal=True)
    assert f == B * H * _fwd_expected(T, True, d), (f, T)
    assert b == 4 * B * H * _tri(T), (b, T)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_noncausal_visits_every_tile(d):
    B, H, T = 2, 2, 5
    f, b = _fwd_bwd_counts(B, H, 128 * T, d, causal=False)
    assert f == B * H * _fwd_expected(T, False, d)
    assert b == 4 * B * H * T * T


def test_causal_skip_at_n4096():
    """N = 4096 (T = 32): 528 of the 1024 tiles of 128 x 128, 48.4% skipped."""
    f, b = _fwd_bwd_counts(1, 1, 4096, 64, causal=True)
    assert f // 4 == 528 and b // 4 == 528
    assert round(100 * (1 - 528 / 1024), 1) == 48.4


@pytest.mark.parametrize("N", [300, 1000, 1100])
def test_ragged_tail_forward(N):
    """A partial last query tile counts in full: the forward at d <= 128
    visits the tiles of T = ceil(N / 128)."""
    T = (N + 127) // 128
    f, _ = _fwd_bwd_counts(1, 2, N, 128, causal=True)
    assert f == 2 * _fwd_expected(T, True, 128)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_visits_kept_blocks_only(d, causal):
    """With a 128 x 128 block mask, exactly the kept (and, causal, visible)
    blocks are computed in each pass (a query tile past the last row keeps
    nothing)."""
    B, H, T = 1, 3, 6
    rng = np.random.default_rng(11 + d + causal)
    bm = rng.random((B * H, T, T)) < 0.4
    bm[:, 2, :] = False  # a query block that keeps nothing
    visible = np.tril(np.ones((T, T), bool)) if causal else np.ones((T, T), bool)
    kept = int((bm & visible[None]).sum())
    f, b = _fwd_bwd_counts(B, H, 128 * T, d, causal, block_mask=bm)
    assert f == 4 * kept and b == 4 * kept, (f, b, kept)


def test_varlen_counts_per_sequence():
    """Packed sequences of 128-multiple lengths (Nq = Nk per sequence): the
    sum over sequences and heads of each sequence's count."""
    lengths = [128, 384, 1024, 640]
    H, d = 2, 128
    q, k, v, do, cu_q, cu_k = varlen_inputs(lengths, lengths, H, d, "bf16", seed=5)
    q, k, v, do, cu_q, cu_k = (x.to(DEV) for x in (q, k, v, do, cu_q, cu_k))
    mx = max(lengths)
    out = {}

    def fwd():
        out["o"], out["lse"] = fa.forward_varlen(q, k, v, cu_q, cu_k, mx, mx, causal=True)

    def bwd():
        fa.backward_varlen(q, k, v, out["o"], out["lse"], do, cu_q, cu_k, mx, mx, causal=True)

    f, _ = _counts(fwd)
    _, b = _counts(bwd)
    assert f == H * sum(_fwd_expected(n // 128, True, d) for n in lengths), f
    assert b == 4 * H * sum(_tri(n // 128) for n in lengths), b

"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these checks retypes the oracle's own formula: each compares it with
a value the page prints, a closed form, an independent algorithm (the online
recurrence, a library log-sum-exp, torch's float64 CPU attention and its
autograd), or finite differences.  ``test_planted_mistakes_are_caught``
shows that a plausible mistake in any building block fails at least one pin.

P3 = the tutorial page "FlashAttention 为什么不需要存下注意力矩阵" (jefxiong.cn).
"""
import os

import numpy as np
import pytest
import scipy.special
import torch

from exact_io_aware_forward_gb300.synth import attention_inputs, page_inputs, as_float64
from oracle import attention as A
from oracle import online as OL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


# ---------------------------------------------------------------- page values
def test_trace_matches_page():
    """P3 section 04.1: m, l and the rescale factor of query 0, block by block."""
    q, k, v = page_inputs(8, 4, 0)
    _, _, trace = OL.online_attention(q, k, v, block=2, trace_row=0)
    want = _rows("trace_query0_rng0.txt")
    assert len(trace) == len(want)
    for (j0, m, l, corr), row in zip(trace, want):
        assert j0 == int(row[0])
        assert round(m, 4) == pytest.approx(float(row[1]), abs=1e-12)
        assert round(l, 4) == pytest.approx(float(row[2]), abs=1e-12)
        assert round(corr, 4) == pytest.approx(float(row[3]), abs=1e-12)


@pytest.mark.parametrize("row", _rows("exactness_table.txt"), ids=lambda r: f"N{r[0]}-{r[2]}")
def test_exactness_table(row):
    """P3 section 04.2: materialised and streamed results agree to float64 rounding."""
    N, D, causal = int(row[0]), int(row[1]), row[2] == "True"
    q, k, v = page_inputs(N, D, N)
    ref, lse_ref = A.forward_head(q, k, v, 1 / np.sqrt(D), causal)
    got, lse_got, _ = OL.online_attention(q, k, v, block=64, causal=causal)
    err = np.abs(ref - got).max()
    # The page's printed errors are all below 1e-15; allow the BLAS-dependent
    # last digits a factor 2.
    assert err < 2e-15, err
    assert np.abs(lse_ref - lse_got).max() < 1e-13


@pytest.mark.parametrize("block", [1, 2, 3, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_online_equals_naive_small_blocks(block, causal):
    """The recurrence holds for any block size, down to one key (P3 section 3.2)."""
    q, k, v = page_inputs(256, 64, 256)
    ref, lse_ref = A.forward_head(q, k, v, 0.125, causal)
    got, lse_got, _ = OL.online_attention(q, k, v, block=block, causal=causal)
    assert np.abs(ref - got).max() < 2e-15
    assert np.abs(lse_ref - lse_got).max() < 1e-13


def test_rescale_ablation_breaks_result():
    """P3 section 09: without the rescale the streamed output is wrong (~0.276)."""
    (N, D, emax, emean), = _rows("rescale_ablation.txt")
    N, D = int(N), int(D)
    q, k, v = page_inputs(N, D, N)
    ref, _ = A.forward_head(q, k, v, 1 / np.sqrt(D), False)
    got, _, _ = OL.online_attention(q, k, v, block=64, rescale=False)
    err = np.abs(ref - got)
    assert float(f"{err.max():.3g}") == float(emax)
    assert float(f"{err.mean():.3g}") == float(emean)


def test_causal_block_count():
    """P3 section 04.5: 2080 of 4096 blocks kept, 49.2% skipped; T(T+1)/2 in general."""
    (N, Bk, total, kept, pct), = _rows("causal_blocks.txt")
    N, Bk = int(N), int(Bk)
    got = OL.causal_blocks_kept(N, Bk, Bk)
    assert (N // Bk) ** 2 == int(total)
    assert got == int(kept)
    assert round(100 * (1 - got / int(total)), 1) == float(pct)
    for T in (1, 2, 5, 17, 64):
        assert OL.causal_blocks_kept(T * 128, 128, 128) == T * (T + 1) // 2


# --------------------------------------------------------------- closed forms
def test_uniform_scores_give_mean_of_v():
    """Q = 0 makes every score 0: O is the mean of the visible V rows, LSE = log(count)."""
    rng = np.random.default_rng(7)
    N, d = 37, 8
    q = np.zeros((N, d))
    k = rng.normal(size=(N, d))
    v = rng.normal(size=(N, d))
    o, lse = A.forward_head(q, k, v, 0.3, causal=False)
    assert np.allclose(o, v.mean(axis=0)[None, :], atol=1e-14)
    assert np.allclose(lse, np.log(N), atol=1e-14)
    o, lse = A.forward_head(q, k, v, 0.3, causal=True)
    prefix = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None]
    assert np.allclose(o, prefix, atol=1e-14)
    assert np.allclose(lse, np.log(np.arange(1, N + 1)), atol=1e-14)


def test_causal_row0_and_single_key():
    """Causal row 0 sees only key 0: O_0 = V_0, LSE_0 = s q_0.k_0.  N = 1 likewise."""
    rng = np.random.default_rng(8)
    N, d, s = 19, 16, 0.25
    q, k, v = (rng.normal(size=(N, d)) for _ in range(3))
    o, lse = A.forward_head(q, k, v, s, causal=True)
    assert np.allclose(o[0], v[0], atol=1e-15)
    assert lse[0] == pytest.approx(s * q[0] @ k[0], abs=1e-14)
    o1, lse1 = A.forward_head(q[:1], k[:1], v[:1], s, causal=False)
    assert np.allclose(o1, v[:1], atol=1e-15)
    dq, dk, dv = A.backward_head(q[:1], k[:1], v[:1], v[:1] * 0 + 1.5, s, False)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0
    assert np.allclose(dv, 1.5)


def test_probabilities_rows_sum_to_one_and_lse_independent():
    rng = np.random.default_rng(9)
    N, d, s = 50, 12, 0.4
    q, k, v = (rng.normal(size=(N, d)) * 3 for _ in range(3))
    for causal in (False, True):
        p = A.probabilities_head(q, k, s, causal)
        assert np.allclose(p.sum(axis=1), 1.0, atol=1e-14)
        if causal:
            assert np.all(np.triu(p, 1) == 0)
        _, lse = A.forward_head(q, k, v, s, causal)
        sc = s * q @ k.T
        if causal:
            sc = np.where(np.triu(np.ones((N, N), bool), 1), -np.inf, sc)
        assert np.allclose(lse, scipy.special.logsumexp(sc, axis=1), atol=1e-13)


# ------------------------------------------------------- library cross-checks
def _torch_reference(q, k, v, do, scale, causal):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    out.backward(torch.tensor(do, dtype=torch.float64))
    return out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 8), (7, 4), (64, 16), (129, 32)])
def test_against_torch_float64(causal, N, d):
    """Forward and gradients equal torch's float64 CPU attention + autograd."""
    q, k, v, do = as_float64(*attention_inputs(2, 3, N, d, "bf16", seed=N + d))
    scale = 1.0 / np.sqrt(d)
    o, lse = A.forward(q, k, v, scale, causal)
    dq, dk, dv = A.backward(q, k, v, do, scale, causal)
    to, tdq, tdk, tdv = _torch_reference(q, k, v, do, scale, causal)
    assert np.abs(o - to).max() < 1e-12
    for g, t in ((dq, tdq), (dk, tdk), (dv, tdv)):
        assert np.abs(g - t).max() < 1e-11


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    """Central differences of L = sum(dO * O) on tiny inputs (N <= 16, d <= 8)."""
    rng = np.random.default_rng(11 + causal)
    N, d, s, h = 9, 5, 0.7, 1e-6
    q, k, v, do = (rng.normal(size=(N, d)) for _ in range(4))
    dq, dk, dv = A.backward_head(q, k, v, do, s, causal)

    def loss(qq, kk, vv):
        return float((A.forward_head(qq, kk, vv, s, causal)[0] * do).sum())

    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for i in range(N):
            for c in range(d):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][i, c] += h
                args_m[which][i, c] -= h
                num[i, c] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        rel = np.linalg.norm(num - grad) / np.linalg.norm(grad)
        assert rel < 1e-7, (which, rel)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    """From rowsum(P) = 1 (P3 section 3.3): sum_j dS_ij = 0, sum_j dK_j = 0,
    sum_j dV_j = sum_i dO_i."""
    rng = np.random.default_rng(12)
    N, d, s = 40, 8, 0.5
    q, k, v, do = (rng.normal(size=(N, d)) for _ in range(4))
    p = A.probabilities_head(q, k, s, causal)
    ds = A._softmax_backward(p, do @ v.T)
    assert np.abs(ds.sum(axis=1)).max() < 1e-13
    dq, dk, dv = A.backward_head(q, k, v, do, s, causal)
    assert np.abs(dk.sum(axis=0)).max() < 1e-12
    assert np.allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)


def test_sampled_backward_equals_full():
    """The striped, sampled backward is the same definition as the full one."""
    rng = np.random.default_rng(13)
    N, d, s = 300, 16, 0.25
    q, k, v, do = (rng.normal(size=(N, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = A.backward_head(q, k, v, do, s, causal)
        rows = np.array([0, 1, 77, 150, 299])
        cols = np.array([0, 5, 128, 298, 299])
        sq, sk, sv = A.backward_head_sampled(q, k, v, do, s, causal, rows, cols, stripe=64)
        assert np.abs(sq - dq[rows]).max() < 1e-13
        assert np.abs(A.backward_head_rows(q, k, v, do, s, causal, rows[::-1]) - dq[rows[::-1]]).max() < 1e-13
        assert np.abs(sk - dk[cols]).max() < 1e-13
        assert np.abs(sv - dv[cols]).max() < 1e-13
        o, lse = A.forward_head(q, k, v, s, causal)
        o2, lse2 = A.forward_head(q, k, v, s, causal, rows=rows)
        assert np.abs(o2 - o[rows]).max() < 1e-15 and np.abs(lse2 - lse[rows]).max() < 1e-14


# ------------------------------------------------------- planted mistakes
def _pins_pass():
    """Run the library cross-check and the finite-difference pin; True if both pass."""
    q, k, v, do = as_float64(*attention_inputs(1, 2, 12, 4, "bf16", seed=5))
    scale = 0.5
    ok = True
    for causal in (False, True):
        o, _ = A.forward(q, k, v, scale, causal)
        dq, dk, dv = A.backward(q, k, v, do, scale, causal)
        to, tdq, tdk, tdv = _torch_reference(q, k, v, do, scale, causal)
        ok &= np.abs(o - to).max() < 1e-12
        for g, t in ((dq, tdq), (dk, tdk), (dv, tdv)):
            ok &= np.abs(g - t).max() < 1e-11
    return bool(ok)


MUTANTS = {
    "dS without the row-sum term": ("_softmax_backward", lambda p, a: p * a),
    "dS with the sign of the row-sum flipped":
        ("_softmax_backward", lambda p, a: p * (a + (a * p).sum(axis=1, keepdims=True))),
    "row sum over the wrong axis":
        ("_softmax_backward", lambda p, a: p * (a - (a * p).sum(axis=0, keepdims=True))),
    "scores without the scale":
        ("_scores", lambda q, k, scale, causal, rows=None, block_mask=None:
         A.__dict__["_orig_scores"](q, k, 1.0, causal, rows, block_mask)),
    "causal mask shifted by one":
        ("_scores", lambda q, k, scale, causal, rows=None, block_mask=None: _shifted_mask(q, k, scale, causal, rows)),
    "softmax without the normalisation":
        ("_softmax_rows", lambda s: (np.exp(s - s.max(axis=1)[:, None]), s.max(axis=1), np.ones(s.shape[0]))),
}


def _shifted_mask(q, k, scale, causal, rows):
    if rows is None:
        rows = np.arange(q.shape[0])
    s = scale * (q[rows] @ k.T)
    if causal:
        keys = np.arange(k.shape[0])
        s = np.where(keys[None, :] >= rows[:, None] + 2, -np.inf, s)
    return s


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    assert _pins_pass()
    attr, bad = MUTANTS[name]
    monkeypatch.setitem(A.__dict__, "_orig_scores", A._scores)
    monkeypatch.setattr(A, attr, bad)
    assert not _pins_pass(), f"pin missed: {name}"


# ------------------------------------------------ fewer queries than keys
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 37), (5, 37), (16, 300)])
def test_rectangular_against_torch(causal, Nq, Nk):
    """Nq <= Nk: torch float64 SDPA with an explicit mask (queries are the last
    Nq positions, so query i sees keys j <= i + Nk - Nq)."""
    rng = np.random.default_rng(Nq * 1000 + Nk)
    d, s = 16, 0.3
    q = rng.normal(size=(Nq, d))
    k, v, = rng.normal(size=(Nk, d)), rng.normal(size=(Nk, d))
    o, lse = A.forward_head(q, k, v, s, causal)
    mask = None
    if causal:
        mask = torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)
    to = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None], torch.tensor(k)[None], torch.tensor(v)[None], attn_mask=mask, scale=s)[0]
    assert np.abs(o - to.numpy()).max() < 1e-12
    full = s * q @ k.T
    if causal:
        full = np.where(mask.numpy(), full, -np.inf)
    assert np.allclose(lse, scipy.special.logsumexp(full, axis=1), atol=1e-13)
    # The last query sees every key: the mask does not change its row.
    o_nc, _ = A.forward_head(q, k, v, s, False)
    assert np.abs(o[-1] - o_nc[-1]).max() < 1e-14
    # The streamed recurrence agrees for any key block size.
    for block in (1, 7, 64):
        so, slse, _ = OL.online_attention(q, k, v, block, scale=s, causal=causal)
        assert np.abs(so - o).max() < 2e-15 and np.abs(slse - lse).max() < 1e-13


def test_key_splits_combine_by_lse():
    """Attention over a key range split in parts equals the LSE-weighted
    combination of the parts: O = sum_s exp(LSE_s - LSE) O_s, LSE = log sum_s exp(LSE_s)."""
    rng = np.random.default_rng(3)
    Nq, Nk, d, s = 4, 1000, 32, 0.2
    q, k, v = rng.normal(size=(Nq, d)), rng.normal(size=(Nk, d)), rng.normal(size=(Nk, d))
    o, lse = A.forward_head(q, k, v, s, False)
    parts = [(0, 130), (130, 131), (131, 600), (600, 1000)]
    lses = np.stack([A.forward_head(q, k[a:b], v[a:b], s, False)[1] for a, b in parts])
    outs = np.stack([A.forward_head(q, k[a:b], v[a:b], s, False)[0] for a, b in parts])
    comb_lse = scipy.special.logsumexp(lses, axis=0)
    comb_o = (np.exp(lses - comb_lse)[:, :, None] * outs).sum(axis=0)
    assert np.abs(comb_lse - lse).max() < 1e-13 and np.abs(comb_o - o).max() < 1e-14


# ------------------------------------------------ block-sparse masks
def _random_block_mask(Tq, Tk, rng, density=0.5, full_rows=True):
    bm = rng.random((Tq, Tk)) < density
    if full_rows:  # every query block keeps at least one key block
        bm[np.arange(Tq), rng.integers(0, Tk, Tq)] = True
    return bm


def test_block_mask_all_ones_is_dense_and_causal_pattern_is_causal():
    rng = np.random.default_rng(21)
    N, d, s = 300, 8, 0.4
    q, k, v, do = (rng.normal(size=(N, d)) for _ in range(4))
    T = (N + 127) // 128
    ones = np.ones((T, T), bool)
    for causal in (False, True):
        o1, l1 = A.forward_head(q, k, v, s, causal)
        o2, l2 = A.forward_head(q, k, v, s, causal, block_mask=ones)
        assert np.abs(o1 - o2).max() == 0 and np.abs(l1 - l2).max() == 0
    tri = np.tril(ones)  # blocks above the diagonal are fully masked by causality anyway
    o1, l1 = A.forward_head(q, k, v, s, True)
    o2, l2 = A.forward_head(q, k, v, s, True, block_mask=tri)
    assert np.abs(o1 - o2).max() == 0
    g1 = A.backward_head(q, k, v, do, s, True)
    g2 = A.backward_head(q, k, v, do, s, True, block_mask=tri)
    assert all(np.abs(a - b).max() == 0 for a, b in zip(g1, g2))


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_against_torch(causal):
    """Random block masks = torch float64 SDPA + autograd with the expanded element mask."""
    rng = np.random.default_rng(22 + causal)
    N, d, s = 400, 16, 0.3
    T = (N + 127) // 128
    bm = _random_block_mask(T, T, rng)
    if causal:
        bm[np.arange(T), np.arange(T)] = True  # every row keeps its diagonal block
    q, k, v, do = (rng.normal(size=(N, d)) for _ in range(4))
    o, lse = A.forward_head(q, k, v, s, causal, block_mask=bm)
    dq, dk, dv = A.backward_head(q, k, v, do, s, causal, block_mask=bm)
    elem = np.kron(bm, np.ones((128, 128), bool))[:N, :N]
    if causal:
        elem &= np.tril(np.ones((N, N), bool))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(elem), scale=s)
    to.backward(torch.tensor(do))
    assert np.abs(o - to.detach().numpy()).max() < 1e-12
    for g, t in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.abs(g - t.numpy()).max() < 1e-11
    full = np.where(elem, s * q @ k.T, -np.inf)
    assert np.allclose(lse, scipy.special.logsumexp(full, axis=1), atol=1e-12)
    # Streaming only over the kept key blocks gives the same rows (P3 section 3.2 for any block order).
    for qb in range(T):
        rows = np.arange(qb * 128, min(N, qb * 128 + 128))
        keys = np.concatenate([np.arange(kb * 128, min(N, kb * 128 + 128)) for kb in range(T) if bm[qb, kb]])
        ref_o, ref_l = A.forward_head(q, k, v, s, causal, rows=rows, block_mask=bm)
        if not causal:
            so, sl, _ = OL.online_attention(q[rows], k[keys], v[keys], 64, scale=s)
            assert np.abs(so - ref_o).max() < 2e-15 and np.abs(sl - ref_l).max() < 1e-13


def test_rows_without_visible_keys():
    """Reading for an empty softmax: O = 0, LSE = -inf, and no gradient."""
    rng = np.random.default_rng(23)
    N, d, s = 260, 8, 0.5
    q, k, v, do = (rng.normal(size=(N, d)) for _ in range(4))
    bm = np.array([[True, False, True], [False, False, False], [False, True, True]])
    o, lse = A.forward_head(q, k, v, s, False, block_mask=bm)
    assert np.all(o[128:256] == 0) and np.all(np.isneginf(lse[128:256]))
    assert np.all(np.isfinite(lse[:128])) and np.all(np.isfinite(lse[256:]))
    dq, dk, dv = A.backward_head(q, k, v, do, s, False, block_mask=bm)
    assert np.all(dq[128:256] == 0)
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))

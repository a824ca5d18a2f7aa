"""Pins of the dropout oracle (no GPU).

The generator is pinned by its published known-answer values, the mapping of
counters to attention entries by a per-entry scalar evaluation, the keep
decisions by binomial bounds, and the dropout algebra by torch float64
autograd with the keep mask given as a constant.
"""
import os

import numpy as np
import pytest
import torch

from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
from oracle import attention as A
from oracle import dropout as DR

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat(), ids=["zeros", "ones", "pi"])
def test_philox_known_answers(row):
    out = DR.philox4x32_10(np.array(row[:4]), row[4:6])
    assert [int(x) for x in out] == row[6:]


def test_philox_batched_equals_single_calls():
    rng = np.random.default_rng(0)
    ctr = rng.integers(0, 2**32, size=(5, 3, 4), dtype=np.uint64)
    key = (0x12345678, 0x9ABCDEF0)
    out = DR.philox4x32_10(ctr, key)
    for idx in np.ndindex(5, 3):
        assert np.array_equal(out[idx], DR.philox4x32_10(ctr[idx], key))


def _draw_scalar(seed, offset, bh, i, j):
    """One entry's 8-bit draw, spelled out from the counter reading."""
    word = DR.philox4x32_10(np.array([j // 16, i, bh, offset]), (seed % 2**32, seed // 2**32))[(j // 4) % 4]
    return (int(word) >> (8 * (j % 4))) & 0xFF


@pytest.mark.parametrize("Nq,Nk,bh,offset", [(5, 19, 3, 7), (3, 16, 0, 0), (2, 49, 17, 2**32 - 1)])
def test_draws_match_per_entry_definition(Nq, Nk, bh, offset):
    seed = 0x0123456789ABCDEF
    got = DR.draws8(seed, offset, bh, np.arange(Nq), Nk)
    for i in range(Nq):
        for j in range(Nk):
            assert got[i, j] == _draw_scalar(seed, offset, bh, i, j), (i, j)


def test_rows_argument_selects_rows():
    full = DR.keep_mask(5, 1, 0.3, 2, 40, 50)
    rows = np.array([39, 0, 17])
    assert np.array_equal(DR.keep_mask(5, 1, 0.3, 2, 40, 50, rows=rows), full[rows])


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_fraction_is_binomial(p):
    """Over 2^20 entries the kept fraction is within 6 sigma of 1 - t/256,
    and different heads, offsets and seeds give different masks."""
    m = DR.keep_mask(42, 3, p, 1, 1024, 1024)
    q = 1.0 - DR.threshold(p) / 256.0
    n = m.size
    assert abs(m.mean() - q) < 6 * np.sqrt(q * (1 - q) / n)
    for other in (DR.keep_mask(42, 3, p, 2, 1024, 1024), DR.keep_mask(42, 4, p, 1, 1024, 1024),
                  DR.keep_mask(43, 3, p, 1, 1024, 1024)):
        agree = (other == m).mean()
        assert abs(agree - (q * q + (1 - q) * (1 - q))) < 0.01


def test_draws_are_uniform_8_bit():
    """Chi-square over the 256 values of the 8-bit draws (2^20 draws), and
    over the 16 byte positions of a generator call."""
    d = DR.draws8(7, 0, 0, np.arange(1024), 1024)
    assert d.max() < 256
    for pos in range(16):  # each byte of the four output words on its own
        col = d[:, pos::16].ravel()
        assert abs(col.mean() - 127.5) < 6 * np.sqrt((256**2 - 1) / 12 / col.size)
    d = d.ravel()
    counts = np.bincount(d, minlength=256)
    e = d.size / 256
    chi2 = ((counts - e) ** 2 / e).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)


def test_threshold_and_scale():
    assert DR.threshold(0.0) == 0 and DR.keep_scale(0.0) == 1.0
    assert DR.threshold(0.5) == 128 and DR.keep_scale(0.5) == 2.0
    assert DR.threshold(0.1) == 26 and DR.keep_scale(0.1) == 256.0 / 230.0
    assert DR.threshold(0.25) == 64 and DR.keep_scale(0.25) == 256.0 / 192.0
    for bad in (-0.1, 1.0, 1.0 - 2**-10):
        with pytest.raises(ValueError):
            DR.threshold(bad)


# ------------------------------------------------------- dropout algebra
def _torch_dropout(q, k, v, do, scale, causal, keep, c):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = scale * tq @ tk.T
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(s.shape, dtype=torch.bool), 1), float("-inf"))
    p = torch.softmax(s, dim=-1)
    out = (p * torch.tensor(keep, dtype=torch.float64) * c) @ tv
    out.backward(torch.tensor(do, dtype=torch.float64))
    return out.detach().numpy(), torch.logsumexp(s, dim=-1).detach().numpy(), tq.grad.numpy(), \
        tk.grad.numpy(), tv.grad.numpy()


def _oracle_dropout(q, k, v, do, scale, causal, keep, c):
    o, lse = A.forward_head(q, k, v, scale, causal, keep=keep, keep_scale=c)
    return (o, lse) + A.backward_head(q, k, v, do, scale, causal, keep=keep, keep_scale=c)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,p", [(7, 4, 0.5), (64, 16, 0.1), (129, 32, 0.3)])
def test_dropout_against_torch_float64(causal, N, d, p):
    q, k, v, do = (x[0, 0] for x in as_float64(*attention_inputs(1, 1, N, d, "bf16", seed=N + d + 1)))
    scale = 1.0 / np.sqrt(d)
    keep = DR.keep_mask(99, 0, p, 0, N, N)
    c = DR.keep_scale(p)
    got = _oracle_dropout(q, k, v, do, scale, causal, keep, c)
    want = _torch_dropout(q, k, v, do, scale, causal, keep, c)
    for g, w in zip(got, want):
        assert np.abs(g - w).max() < 1e-11


def test_all_kept_scale_one_is_plain_attention():
    q, k, v, do = (x[0, 0] for x in as_float64(*attention_inputs(1, 1, 50, 8, "bf16", seed=3)))
    keep = np.ones((50, 50), bool)
    for causal in (False, True):
        o, lse = A.forward_head(q, k, v, 0.3, causal)
        o2, lse2 = A.forward_head(q, k, v, 0.3, causal, keep=keep, keep_scale=1.0)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
        for g, g2 in zip(A.backward_head(q, k, v, do, 0.3, causal),
                         A.backward_head(q, k, v, do, 0.3, causal, keep=keep, keep_scale=1.0)):
            assert np.array_equal(g, g2)


def test_dropout_is_unbiased_on_average():
    """Averaged over many offsets, the dropped output approaches the plain one."""
    q, k, v, _ = (x[0, 0] for x in as_float64(*attention_inputs(1, 1, 16, 4, "bf16", seed=4)))
    o, _ = A.forward_head(q, k, v, 0.5, False)
    p, c = 0.5, DR.keep_scale(0.5)
    acc = np.zeros_like(o)
    n = 2000
    for off in range(n):
        acc += A.forward_head(q, k, v, 0.5, False, keep=DR.keep_mask(1, off, p, 0, 16, 16), keep_scale=c)[0]
    assert np.abs(acc / n - o).max() < 0.1 * np.abs(v).max()


def _dropout_pins_pass():
    q, k, v, do = (x[0, 0] for x in as_float64(*attention_inputs(1, 1, 12, 4, "bf16", seed=8)))
    ok = True
    for causal in (False, True):
        keep = DR.keep_mask(5, 0, 0.4, 0, 12, 12)
        c = DR.keep_scale(0.4)
        for g, w in zip(_oracle_dropout(q, k, v, do, 0.5, causal, keep, c),
                        _torch_dropout(q, k, v, do, 0.5, causal, keep, c)):
            ok &= np.abs(g - w).max() < 1e-11
    return bool(ok)


DROPOUT_MUTANTS = {
    "keep scale not applied": lambda p, keep, c: np.where(keep, p, 0.0),
    "mask inverted": lambda p, keep, c: np.where(keep, 0.0, p * c),
    "scale applied to dropped entries": lambda p, keep, c: np.where(keep, p * c, p * (c - 1.0)),
}


@pytest.mark.parametrize("name", sorted(DROPOUT_MUTANTS))
def test_planted_dropout_mistakes_are_caught(name, monkeypatch):
    assert _dropout_pins_pass()
    monkeypatch.setattr(A, "_dropped", lambda p, keep, c: p if keep is None else DROPOUT_MUTANTS[name](p, keep, c))
    assert not _dropout_pins_pass(), name


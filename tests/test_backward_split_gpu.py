"""The split backward (dQ by a kernel of its own) through its stage entry
points: fa_backward_preprocess with no accumulator, fa_backward_dk_dv and
fa_backward_dq, against the float64 oracle's explicit softmax backward
(relative Frobenius error <= 1e-2), and against the accumulated strategy
(fa_backward_dkdv + fa_backward_dq_convert) on the same inputs.

Sizes span several 128-row tiles with ragged tails, both masks, both 16-bit
types and d in {64, 96, 128}; every head is compared.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
from oracle import attention as A

from gpu_util import GRAD_REL_FRO, rel_fro

pytestmark = pytest.mark.gpu


def _split_backward(q, k, v, do, causal, scale=None):
    """Forward, then the three split stages; returns CPU (dq, dk, dv, delta)."""
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    B, H, N, d = q.shape
    delta = torch.full((B, H, N), float("nan"), device=dev, dtype=torch.float32)
    dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
    fa.fa_backward_preprocess(o, dod, delta, None)
    fa.fa_backward_dk_dv(qd, kd, vd, dod, lse, delta, dk, dv, causal, scale)
    fa.fa_backward_dq(qd, kd, vd, dod, lse, delta, dq, causal, scale)
    fa.fa_device_status()
    return dq.cpu(), dk.cpu(), dv.cpu(), delta.cpu(), o.cpu()


def _check(q, k, v, do, got, causal, scale=None):
    B, H, N, d = q.shape
    s = 1.0 / math.sqrt(d) if scale is None else scale
    qf, kf, vf, dof = as_float64(q, k, v, do)
    g = [x.to(torch.float64).numpy() for x in got[:3]]
    errs = {}
    for i, name in enumerate(("dq", "dk", "dv")):
        gs, rs = [], []
        for b in range(B):
            for h in range(H):
                ref = A.backward_head(qf[b, h], kf[b, h], vf[b, h], dof[b, h], s, causal)
                gs.append(g[i][b, h])
                rs.append(ref[i])
        gn, rn = np.concatenate(gs), np.concatenate(rs)
        assert np.isfinite(gn).all(), name
        if np.linalg.norm(rn) == 0.0:  # one visible key: dS = 0 exactly
            errs[name] = float(np.abs(gn).max())
            assert errs[name] <= 1e-4, (name, errs)
        else:
            errs[name] = rel_fro(gn, rn)
            assert errs[name] <= GRAD_REL_FRO, (name, errs)
    return errs


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 383, 640])
def test_split_stages_match_the_oracle(N, causal, d, dtype):
    q, k, v, do = attention_inputs(1, 2, N, d, dtype, seed=7000 + N + d)
    got = _split_backward(q, k, v, do, causal)
    _check(q, k, v, do, got, causal)
    # D = rowsum(dO * O) of the stored O, from the preprocess stage alone
    o, delta = got[4], got[3]
    want = (do.double() * o.double()).sum(-1)
    assert float((delta.double() - want).abs().max()) <= 1e-3 * float(want.abs().max() + 1)


def test_split_stages_scale_and_wide_scores():
    """A scale other than 1/sqrt(d) and K rows scaled by U(0.5, 3)."""
    q, k, v, do = attention_inputs(2, 3, 700, 128, "bf16", seed=71, k_row_scale=True)
    got = _split_backward(q, k, v, do, True, scale=0.3)
    _check(q, k, v, do, got, True, scale=0.3)


@pytest.mark.parametrize("causal", [False, True])
def test_split_agrees_with_accumulated(causal):
    """Both dQ strategies on the same inputs: the same gradients up to fp32
    summation order (dQ) -- dK and dV differ only in the query tiling."""
    dev = torch.device("cuda:0")
    B, H, N, d = 2, 5, 1100, 128
    q, k, v, do = (x.to(dev) for x in attention_inputs(B, H, N, d, "bf16", seed=77))
    o, lse = fa.forward(q, k, v, causal=causal)
    ws = torch.empty(fa.fa_backward_workspace_size(B, H, N, d), device=dev, dtype=torch.uint8)
    rows = B * H * N
    delta = ws[: rows * 4].view(torch.float32).view(B, H, N)
    off = (rows * 4 + 255) // 256 * 256
    acc = ws[off: off + rows * d * 4].view(torch.float32).view(B, H, N, d)
    a = [torch.empty_like(q) for _ in range(3)]
    fa.fa_backward_preprocess(o, do, delta, acc)
    fa.fa_backward_dkdv(q, k, v, do, lse, delta, acc, a[1], a[2], causal)
    fa.fa_backward_dq_convert(acc, a[0])
    s = [torch.empty_like(q) for _ in range(3)]
    fa.fa_backward_preprocess(o, do, delta, None)
    fa.fa_backward_dk_dv(q, k, v, do, lse, delta, s[1], s[2], causal)
    fa.fa_backward_dq(q, k, v, do, lse, delta, s[0], causal)
    fa.fa_device_status()
    for name, x, y in zip(("dq", "dk", "dv"), a, s):
        err = rel_fro(y.double().cpu().numpy(), x.double().cpu().numpy())
        assert err <= 4e-3, (name, err)


def test_backward_entry_point_takes_the_split_path():
    """fa_backward on dense d = 128 leaves the accumulator region of its
    workspace untouched (the split strategy keeps none) and matches the
    stage-by-stage result bit for bit."""
    dev = torch.device("cuda:0")
    B, H, N, d = 1, 3, 515, 128
    q, k, v, do = (x.to(dev) for x in attention_inputs(B, H, N, d, "bf16", seed=78))
    o, lse = fa.forward(q, k, v, causal=True)
    ws = torch.full((fa.fa_backward_workspace_size(B, H, N, d),), 0xA5, device=dev, dtype=torch.uint8)
    got = [torch.empty_like(q) for _ in range(3)]
    fa.fa_backward(q, k, v, o, do, lse, *got, ws, True)
    rows = B * H * N
    off = (rows * 4 + 255) // 256 * 256
    assert bool((ws[off:] == 0xA5).all())
    ref = _split_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), True)
    for x, y in zip(got, ref[:3]):
        assert torch.equal(x.cpu(), y)


@pytest.mark.parametrize("kind", ["dense64", "dense96", "dense128", "blocksparse", "varlen"])
def test_backward_is_bitwise_reproducible(kind):
    """The split strategy has no atomics: two fa_backward calls on the same
    inputs give the same dQ, dK and dV bit for bit (dense, block-sparse and
    packed layouts; several L2 head groups and ragged tails)."""
    dev = torch.device("cuda:0")
    if kind == "varlen":
        from exact_io_aware_forward_gb300.synth import varlen_inputs
        lq = [700, 129, 2050, 1]
        q, k, v, do, cu_q, cu_k = (x.to(dev) for x in varlen_inputs(lq, lq, 4, 128, "bf16", seed=91))
        L = max(lq)
        o, lse = fa.forward_varlen(q, k, v, cu_q, cu_k, L, L, causal=True)
        run = lambda: fa.backward_varlen(q, k, v, o, lse, do, cu_q, cu_k, L, L, causal=True)  # noqa: E731
    else:
        d = {"dense64": 64, "dense96": 96}.get(kind, 128)
        B, H, N = 2, 24, 1300
        q, k, v, do = (x.to(dev) for x in attention_inputs(B, H, N, d, "bf16", seed=92 + d))
        mask = None
        if kind == "blocksparse":
            T = (N + 127) // 128
            bm = np.random.default_rng(5).random((B * H, T, T)) < 0.6
            bm[:, np.arange(T), np.arange(T)] = True
            mask = torch.from_numpy(bm.astype(np.uint8)).to(dev)
        o, lse = fa.forward(q, k, v, causal=True, block_mask=mask)
        run = lambda: fa.backward(q, k, v, o, lse, do, causal=True, block_mask=mask)  # noqa: E731
    first = [x.clone() for x in run()]
    second = run()
    fa.fa_device_status()
    for name, a, b in zip(("dq", "dk", "dv"), first, second):
        assert torch.equal(a, b), name

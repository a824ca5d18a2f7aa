"""Dropout regenerated from the Philox seed and offset: CUDA path vs the
float64 oracle.

The keep mask is integer work and must match the oracle's generator bit for
bit; O, LSE and the gradients must match the oracle given that mask.  The
backward pass regenerates the mask (nothing is stored between the calls).
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
from oracle import attention as A
from oracle import dropout as DR

from gpu_util import GRAD_REL_FRO, LSE_TOL, O_TOL, rel_fro

pytestmark = pytest.mark.gpu

# Output bound for dropout: kept weights are scaled by 1 / (1 - p), so |O| can
# exceed the range the fixed bf16 / fp16 bounds were set for; the bound is then
# the 16-bit representation floor, one ulp at the largest |O| (2^-8 relative in
# bf16, 2^-11 in fp16).
ULP_REL = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}


@pytest.mark.parametrize("BH,Nq,Nk", [(3, 37, 77), (2, 128, 256), (1, 5, 8)])
@pytest.mark.parametrize("p,seed,offset", [(0.1, 0, 0), (0.5, 0x0123456789ABCDEF, 7), (0.9, 2**40 + 3, 2**32 - 1)])
def test_keep_mask_is_bit_exact(BH, Nq, Nk, p, seed, offset):
    keep = torch.empty((BH, Nq, Nk), device="cuda:0", dtype=torch.uint8)
    fa.fa_dropout_keep_mask(keep, p, seed, offset)
    fa.fa_device_status()
    got = keep.cpu().numpy().astype(bool)
    for bh in range(BH):
        want = DR.keep_mask(seed, offset, p, bh, Nq, Nk)
        assert np.array_equal(got[bh], want), bh


def _run(q, k, v, do, causal, p, seed, offset):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, dropout_p=p, seed=seed, offset=offset)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=causal, dropout_p=p, seed=seed, offset=offset)
    fa.fa_device_status()
    return tuple(x.cpu() for x in (o, lse, dq, dk, dv))


def _check(q, k, v, do, causal, p, seed, offset, o, lse, dq, dk, dv, dtype):
    B, H, N, d = q.shape
    s = 1.0 / math.sqrt(d)
    c = DR.keep_scale(p)
    qf, kf, vf, dof = as_float64(q, k, v, do)
    eo = el = omax = 0.0
    gets = {n: [] for n in ("dq", "dk", "dv")}
    refs = {n: [] for n in ("dq", "dk", "dv")}
    for b in range(B):
        for h in range(H):
            keep = DR.keep_mask(seed, offset, p, b * H + h, N, N)
            ro, rl = A.forward_head(qf[b, h], kf[b, h], vf[b, h], s, causal, keep=keep, keep_scale=c)
            eo = max(eo, float(np.abs(o[b, h].double().numpy() - ro).max()))
            el = max(el, float(np.abs(lse[b, h].double().numpy() - rl).max()))
            omax = max(omax, float(np.abs(ro).max()))
            rg = A.backward_head(qf[b, h], kf[b, h], vf[b, h], dof[b, h], s, causal, keep=keep, keep_scale=c)
            for n, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), rg):
                gets[n].append(g[b, h].double().numpy())
                refs[n].append(r)
    tol = max(O_TOL[dtype], ULP_REL[dtype] * omax)
    assert eo <= tol and el <= LSE_TOL, (eo, tol, el)
    # With one key dS = 0 exactly, so dQ = dK = 0 and no relative error is
    # defined.  The kernel's D = rowsum(dO * O) reads the stored 16-bit O, which
    # under dropout (O = c V) is rounded; the resulting dS is bounded by
    # sum_c |dO_c O_c| times the 16-bit relative rounding, and dQ, dK by that
    # times s max|K| or s max|Q|.
    dslack = 2 * ULP_REL[dtype] * float((np.abs(dof) * np.abs(o.double().numpy())).sum(axis=-1).max())
    for n in gets:
        g, r = np.concatenate(gets[n]), np.concatenate(refs[n])
        if np.linalg.norm(r) < 1e-12:
            other = kf if n == "dq" else qf
            assert np.abs(g).max() <= max(1e-4, s * dslack * float(np.abs(other).max())), n
            continue
        e = rel_fro(g, r)
        assert e <= GRAD_REL_FRO, (n, e)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,dtype,p", [(300, 64, "fp16", 0.1), (640, 128, "bf16", 0.2), (1000, 64, "bf16", 0.5),
                                         (513, 128, "fp16", 0.15), (1, 64, "bf16", 0.3), (450, 96, "bf16", 0.25)])
def test_dropout_matches_oracle(causal, N, d, dtype, p):
    B, H = 1, 3
    q, k, v, do = attention_inputs(B, H, N, d, dtype, seed=5000 + N + d)
    seed, offset = 1234 + N, 3
    out = _run(q, k, v, do, causal, p, seed, offset)
    _check(q, k, v, do, causal, p, seed, offset, *out, dtype)


def test_dropout_two_batches_and_seeds_differ():
    """B = 2 (head index b*H + h in the counter); a new offset gives a new mask,
    the same (seed, offset) gives the same result twice."""
    B, H, N, d = 2, 2, 384, 128
    q, k, v, do = attention_inputs(B, H, N, d, "bf16", seed=61)
    a = _run(q, k, v, do, True, 0.25, 99, 0)
    _check(q, k, v, do, True, 0.25, 99, 0, *a, "bf16")
    b = _run(q, k, v, do, True, 0.25, 99, 0)
    assert torch.equal(a[0], b[0]) and torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    c = _run(q, k, v, do, True, 0.25, 99, 1)
    assert not torch.equal(a[0], c[0])
    assert torch.equal(a[1], c[1])  # LSE does not depend on the mask


def test_dropout_zero_is_plain_attention():
    B, H, N, d = 1, 2, 300, 64
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in attention_inputs(B, H, N, d, "fp16", seed=62))
    o1, l1 = fa.forward(q, k, v, causal=True)
    o2, l2 = fa.forward(q, k, v, causal=True, dropout_p=1e-7, seed=5, offset=0)  # rounds to t = 0
    fa.fa_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_dropout_stages_equal_the_full_call():
    """fa_backward_dropout accumulates dQ: preprocess + fa_backward_dkdv_dropout
    + dq_convert give its result bit for bit.  The split stages
    (fa_backward_dk_dv_dropout + fa_backward_dq_dropout, no accumulator) agree
    within the 16-bit rounding of the two orders."""
    B, H, N, d = 1, 3, 700, 128
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in attention_inputs(B, H, N, d, "bf16", seed=63))
    p, seed, offset = 0.3, 77, 5
    o, lse = fa.forward(q, k, v, dropout_p=p, seed=seed, offset=offset)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, dropout_p=p, seed=seed, offset=offset)
    ws = torch.empty(fa.fa_backward_workspace_size(B, H, N, d), device=dev, dtype=torch.uint8)
    rows = B * H * N
    delta = ws[: rows * 4].view(torch.float32).view(B, H, N)
    off = (rows * 4 + 255) // 256 * 256
    acc = ws[off: off + rows * d * 4].view(torch.float32).view(B, H, N, d)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    fa.fa_backward_preprocess(o, do, delta, acc)
    fa.fa_backward_dkdv_dropout(q, k, v, do, lse, delta, acc, dk2, dv2, p, seed, offset)
    fa.fa_backward_dq_convert(acc, dq2)
    fa.fa_device_status()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert float((dq.float() - dq2.float()).abs().max()) <= 1e-2 * float(dq.float().abs().max())
    dq3, dk3, dv3 = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    fa.fa_backward_dk_dv_dropout(q, k, v, do, lse, delta, dk3, dv3, p, seed, offset)
    fa.fa_backward_dq_dropout(q, k, v, do, lse, delta, dq3, p, seed, offset)
    fa.fa_device_status()
    for x, y in ((dq, dq3), (dk, dk3), (dv, dv3)):
        assert float((x.float() - y.float()).abs().max()) <= 1e-2 * float(x.float().abs().max())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,dtype,p", [(650, 64, "fp16", 0.2), (300, 96, "bf16", 0.5)])
def test_dropout_split_stages_match_oracle(causal, N, d, dtype, p):
    """The split stages alone against the oracle on ragged sizes (B = 2, so the
    head index b * H + h of the generator's counter is exercised)."""
    B, H = 2, 2
    dev = torch.device("cuda:0")
    q, k, v, do = attention_inputs(B, H, N, d, dtype, seed=6100 + N + causal)
    seed, offset = 2**33 + 17, 9
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, dropout_p=p, seed=seed, offset=offset)
    delta = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    fa.fa_backward_preprocess(o, dod, delta, None)
    fa.fa_backward_dk_dv_dropout(qd, kd, vd, dod, lse, delta, dk, dv, p, seed, offset, causal=causal)
    fa.fa_backward_dq_dropout(qd, kd, vd, dod, lse, delta, dq, p, seed, offset, causal=causal)
    fa.fa_device_status()
    out = tuple(x.cpu() for x in (o, lse, dq, dk, dv))
    _check(q, k, v, do, causal, p, seed, offset, *out, dtype)


def test_dropout_split_stages_reject_d256():
    B, H, N, d = 1, 1, 128, 256
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in attention_inputs(B, H, N, d, "bf16", seed=64))
    lse = torch.zeros((B, H, N), device=dev, dtype=torch.float32)
    delta = torch.zeros_like(lse)
    with pytest.raises(fa.FAError):
        fa.fa_backward_dq_dropout(q, k, v, do, lse, delta, torch.empty_like(q), 0.1, 1, 0)

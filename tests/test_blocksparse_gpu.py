"""Block-sparse attention (128 x 128 block mask): CUDA path vs the float64 oracle.

Kept blocks must match the oracle exactly as dense attention does; rows that
keep no key get O = 0, LSE = -inf and dQ = 0; an all-ones mask must give the
dense kernels' result bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
from oracle import attention as A

from gpu_util import GRAD_REL_FRO, LSE_TOL, O_TOL, rel_fro

pytestmark = pytest.mark.gpu


def _mask(heads, N, density, seed, causal, empty_block_row=None):
    T = (N + 127) // 128
    rng = np.random.default_rng(seed)
    bm = rng.random((heads, T, T)) < density
    bm[:, np.arange(T), np.arange(T)] = True  # every query block keeps its diagonal block
    if empty_block_row is not None:
        bm[:, empty_block_row, :] = False
    return bm


def _run(q, k, v, do, bm, causal):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    md = torch.from_numpy(bm.astype(np.uint8)).to(dev)
    o, lse = fa.forward(qd, kd, vd, causal=causal, block_mask=md)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=causal, block_mask=md)
    fa.fa_device_status()
    return tuple(x.cpu() for x in (o, lse, dq, dk, dv))


def _check(q, k, v, do, bm, causal, o, lse, dq, dk, dv, dtype):
    B, H, N, d = q.shape
    s = 1.0 / math.sqrt(d)
    qf, kf, vf, dof = as_float64(q, k, v, do)
    eo = el = 0.0
    gets = {n: [] for n in ("dq", "dk", "dv")}
    refs = {n: [] for n in ("dq", "dk", "dv")}
    for b in range(B):
        for h in range(H):
            m = bm[0 if bm.shape[0] == 1 else b * H + h]
            ro, rl = A.forward_head(qf[b, h], kf[b, h], vf[b, h], s, causal, block_mask=m)
            gl = lse[b, h].double().numpy()
            assert np.array_equal(np.isneginf(gl), np.isneginf(rl))
            fin = np.isfinite(rl)
            eo = max(eo, float(np.abs(o[b, h].double().numpy() - ro).max()))
            if fin.any():
                el = max(el, float(np.abs(gl[fin] - rl[fin]).max()))
            rg = A.backward_head(qf[b, h], kf[b, h], vf[b, h], dof[b, h], s, causal, block_mask=m)
            for n, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), rg):
                gets[n].append(g[b, h].double().numpy())
                refs[n].append(r)
    assert eo <= O_TOL[dtype] and el <= LSE_TOL, (eo, el)
    for n in gets:
        e = rel_fro(np.concatenate(gets[n]), np.concatenate(refs[n]))
        assert e <= GRAD_REL_FRO, (n, e)


@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,dtype", [(300, 64, "fp16"), (640, 128, "bf16"), (1000, 64, "bf16"), (513, 128, "fp16"),
                                       (700, 96, "bf16")])
def test_blocksparse_matches_oracle(per_head, causal, N, d, dtype):
    B, H = 1, 3
    q, k, v, do = attention_inputs(B, H, N, d, dtype, seed=3000 + N + d)
    bm = _mask(B * H if per_head else 1, N, 0.45, seed=N + causal, causal=causal)
    o, lse, dq, dk, dv = _run(q, k, v, do, bm, causal)
    _check(q, k, v, do, bm, causal, o, lse, dq, dk, dv, dtype)


def test_blocksparse_empty_rows():
    """A query block that keeps nothing: O = 0, LSE = -inf, dQ = 0; a key block kept by
    nobody gets dK = dV = 0."""
    B, H, N, d = 1, 2, 520, 128
    q, k, v, do = attention_inputs(B, H, N, d, "bf16", seed=77)
    T = (N + 127) // 128
    bm = np.ones((1, T, T), bool)
    bm[0, 1, :] = False  # query block 1 keeps no key block
    bm[0, :, 3] = False  # key block 3 is kept by no query block
    o, lse, dq, dk, dv = _run(q, k, v, do, bm, False)
    assert torch.all(o[:, :, 128:256] == 0) and torch.all(torch.isneginf(lse[:, :, 128:256]))
    assert torch.all(dq[:, :, 128:256] == 0)
    assert torch.all(dk[:, :, 384:512] == 0) and torch.all(dv[:, :, 384:512] == 0)
    _check(q, k, v, do, bm, False, o, lse, dq, dk, dv, "bf16")


@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_all_ones_equals_dense(causal):
    B, H, N, d = 2, 2, 700, 128
    q, k, v, do = attention_inputs(B, H, N, d, "bf16", seed=78)
    T = (N + 127) // 128
    o, lse, dq, dk, dv = _run(q, k, v, do, np.ones((1, T, T), bool), causal)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o2, lse2 = fa.forward(qd, kd, vd, causal=causal)
    dq2, dk2, dv2 = fa.backward(qd, kd, vd, o2, lse2, dod, causal=causal)
    fa.fa_device_status()
    assert torch.equal(o, o2.cpu()) and torch.equal(lse, lse2.cpu())
    # both take the split backward (dQ by its own kernel, no atomics)
    assert torch.equal(dk, dk2.cpu()) and torch.equal(dv, dv2.cpu()) and torch.equal(dq, dq2.cpu())


def test_blocksparse_stages_equal_the_full_call():
    """fa_backward_blocksparse takes the split backward: preprocess without an
    accumulator + fa_backward_dk_dv_blocksparse + fa_backward_dq_blocksparse
    (the launches the benchmark times one by one) give its result bit for bit,
    and the accumulator region of its workspace stays untouched.  The
    accumulated stages (fa_backward_dkdv_blocksparse + dq_convert) agree."""
    B, H, N, d = 1, 4, 1100, 128
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in attention_inputs(B, H, N, d, "bf16", seed=79))
    md = torch.from_numpy(_mask(B * H, N, 0.4, seed=5, causal=False).astype(np.uint8)).to(dev)
    o, lse = fa.forward(q, k, v, block_mask=md)
    ws = torch.full((fa.fa_backward_workspace_size(B, H, N, d),), 0xA5, device=dev, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    fa.fa_backward_blocksparse(q, k, v, o, do, lse, dq, dk, dv, md, ws)
    rows = B * H * N
    off = (rows * 4 + 255) // 256 * 256
    assert bool((ws[off:] == 0xA5).all())
    delta = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    fa.fa_backward_preprocess(o, do, delta, None)
    fa.fa_backward_dk_dv_blocksparse(q, k, v, do, lse, delta, dk2, dv2, md)
    fa.fa_backward_dq_blocksparse(q, k, v, do, lse, delta, dq2, md)
    fa.fa_device_status()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2) and torch.equal(dq, dq2)
    acc = torch.empty((B, H, N, d), device=dev, dtype=torch.float32)
    dq3, dk3, dv3 = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    fa.fa_backward_preprocess(o, do, delta, acc)
    fa.fa_backward_dkdv_blocksparse(q, k, v, do, lse, delta, acc, dk3, dv3, md)
    fa.fa_backward_dq_convert(acc, dq3)
    fa.fa_device_status()
    for x, y in ((dq, dq3), (dk, dk3), (dv, dv3)):
        assert float((x.float() - y.float()).abs().max()) <= 1e-2 * float(x.float().abs().max())


@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_split_stages_on_ragged_sizes(causal):
    """The split stages alone against the oracle on a ragged size with
    per-head masks, an empty query block and an unkept key block."""
    B, H, N, d = 1, 3, 650, 64
    dev = torch.device("cuda:0")
    q, k, v, do = attention_inputs(B, H, N, d, "fp16", seed=81 + causal)
    bm = _mask(B * H, N, 0.5, seed=9, causal=causal)
    bm[:, 3, :] = False
    bm[:, :, 1] = False
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    md = torch.from_numpy(bm.astype(np.uint8)).to(dev)
    o, lse = fa.forward(qd, kd, vd, causal=causal, block_mask=md)
    delta = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    fa.fa_backward_preprocess(o, dod, delta, None)
    fa.fa_backward_dk_dv_blocksparse(qd, kd, vd, dod, lse, delta, dk, dv, md, causal)
    fa.fa_backward_dq_blocksparse(qd, kd, vd, dod, lse, delta, dq, md, causal)
    fa.fa_device_status()
    _check(q, k, v, do, bm, causal, o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu(), "fp16")

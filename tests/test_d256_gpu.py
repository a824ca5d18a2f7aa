"""Head dimension 256: CUDA path vs the float64 oracle, dense and packed, with
and without dropout (block masks are not supported at this width)."""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs, varlen_inputs
from oracle import attention as A
from oracle import dropout as DR
from oracle import varlen as VL

from gpu_util import GRAD_REL_FRO, LSE_TOL, O_TOL, rel_fro

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
D = 256


def _check_dense(q, k, v, o, lse, causal, dtype, keep_fn=None, c=1.0, o_tol=None):
    B, H, N, _ = q.shape
    qf, kf, vf = as_float64(q, k, v)
    s = 1.0 / math.sqrt(D)
    eo = el = 0.0
    for b in range(B):
        for h in range(H):
            keep = keep_fn(b * H + h) if keep_fn else None
            ro, rl = A.forward_head(qf[b, h], kf[b, h], vf[b, h], s, causal, keep=keep, keep_scale=c)
            eo = max(eo, float(np.abs(o[b, h].double().cpu().numpy() - ro).max()))
            el = max(el, float(np.abs(lse[b, h].double().cpu().numpy() - rl).max()))
    assert eo <= (o_tol or O_TOL[dtype]) and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,dtype", [(1, "bf16"), (63, "fp16"), (300, "bf16"), (777, "fp16"), (1024, "bf16")])
def test_d256_dense_forward(causal, N, dtype):
    B, H = 1, 2
    q, k, v, _ = attention_inputs(B, H, N, D, dtype, seed=256 + N)
    o, lse = fa.forward(*(x.to(DEV) for x in (q, k, v)), causal=causal)
    fa.fa_device_status()
    _check_dense(q, k, v, o, lse, causal, dtype)


def test_d256_dropout_forward():
    B, H, N, p, seed, off = 2, 2, 500, 0.25, 9, 2
    q, k, v, _ = attention_inputs(B, H, N, D, "bf16", seed=257)
    o, lse = fa.forward(*(x.to(DEV) for x in (q, k, v)), causal=True, dropout_p=p, seed=seed, offset=off)
    fa.fa_device_status()
    _check_dense(q, k, v, o, lse, True, "bf16", keep_fn=lambda bh: DR.keep_mask(seed, off, p, bh, N, N),
                 c=DR.keep_scale(p), o_tol=max(O_TOL["bf16"], 2.0 ** -8 * float(v.abs().max()) / (1 - p)))


@pytest.mark.parametrize("causal", [False, True])
def test_d256_varlen_forward(causal):
    lq, lk = [130, 1, 400, 0], [200, 64, 399, 17]
    q, k, v, _, cu_q, cu_k = varlen_inputs(lq, lk, 2, D, "bf16", seed=258, with_do=False)
    o, lse = fa.forward_varlen(*(x.to(DEV) for x in (q, k, v, cu_q, cu_k)), max(lq), max(lk), causal=causal)
    fa.fa_device_status()
    ro, rl = VL.forward_varlen(*as_float64(q, k, v), cu_q.numpy(), cu_k.numpy(), 1 / 16.0, causal)
    assert float(np.abs(o.double().cpu().numpy() - ro).max()) <= O_TOL["bf16"]
    gl = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert float(np.abs(gl[fin] - rl[fin]).max()) <= LSE_TOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,dtype", [(1, "bf16"), (200, "fp16"), (513, "bf16")])
def test_d256_backward(causal, N, dtype):
    B, H = 1, 2
    q, k, v, do = attention_inputs(B, H, N, D, dtype, seed=260 + N)
    dev = [x.to(DEV) for x in (q, k, v, do)]
    o, lse = fa.forward(*dev[:3], causal=causal)
    dq, dk, dv = fa.backward(*dev[:3], o, lse, dev[3], causal=causal)
    fa.fa_device_status()
    qf, kf, vf, dof = as_float64(q, k, v, do)
    s = 1.0 / math.sqrt(D)
    for h in range(H):
        ref = A.backward_head(qf[0, h], kf[0, h], vf[0, h], dof[0, h], s, causal)
        for g, r in zip((dq, dk, dv), ref):
            g = g[0, h].double().cpu().numpy()
            if np.linalg.norm(r) < 1e-12:
                assert np.abs(g).max() <= 1e-4
            else:
                assert rel_fro(g, r) <= GRAD_REL_FRO


def test_d256_varlen_backward_with_dropout():
    lq, lk = [130, 300], [200, 300]
    q, k, v, do, cu_q, cu_k = varlen_inputs(lq, lk, 2, D, "bf16", seed=261)
    dev = [x.to(DEV) for x in (q, k, v, do, cu_q, cu_k)]
    p, seed, off = 0.2, 5, 1
    o, lse = fa.forward_varlen(*dev[:3], dev[4], dev[5], 300, 300, causal=True, dropout_p=p, seed=seed, offset=off)
    dq, dk, dv = fa.backward_varlen(*dev[:3], o, lse, dev[3], dev[4], dev[5], 300, 300, causal=True, dropout_p=p,
                                    seed=seed, offset=off)
    fa.fa_device_status()
    qf, kf, vf, dof = as_float64(q, k, v, do)
    c = DR.keep_scale(p)
    cq, ck = cu_q.numpy(), cu_k.numpy()
    for b in range(2):
        for h in range(2):
            keep = DR.keep_mask(seed, off, p, b * 2 + h, cq[b + 1] - cq[b], ck[b + 1] - ck[b])
            args = (qf[cq[b]:cq[b + 1], h], kf[ck[b]:ck[b + 1], h], vf[ck[b]:ck[b + 1], h])
            ref = A.backward_head(*args, dof[cq[b]:cq[b + 1], h], 1 / 16.0, True, keep=keep, keep_scale=c)
            got = (dq[cq[b]:cq[b + 1], h], dk[ck[b]:ck[b + 1], h], dv[ck[b]:ck[b + 1], h])
            for g, r in zip(got, ref):
                assert rel_fro(g.double().cpu().numpy(), r) <= GRAD_REL_FRO


def test_d256_block_mask_is_unsupported():
    q, k, v, do = (x.to(DEV) for x in attention_inputs(1, 1, 128, D, "bf16", seed=259))
    md = torch.ones((1, 1, 1), dtype=torch.uint8, device=DEV)
    with pytest.raises(fa.FAError) as e:
        fa.forward(q, k, v, block_mask=md)
    assert e.value.code == 2
    fa.fa_device_status()

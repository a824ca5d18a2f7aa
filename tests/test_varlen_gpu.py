"""Packed variable-length batches (bottom-right causal per sequence, Nq != Nk,
empty ranges) and head dimension 96: CUDA path vs the float64 oracle."""
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


def _run_varlen(q, k, v, do, cu_q, cu_k, lq, lk, causal, p=0.0, seed=0, offset=0):
    qd, kd, vd, dod, cqd, ckd = (x.to(DEV) for x in (q, k, v, do, cu_q, cu_k))
    mq, mk = max(max(lq), 1), max(max(lk), 1)
    o, lse = fa.forward_varlen(qd, kd, vd, cqd, ckd, mq, mk, causal=causal, dropout_p=p, seed=seed, offset=offset)
    dq, dk, dv = fa.backward_varlen(qd, kd, vd, o, lse, dod, cqd, ckd, mq, mk, causal=causal, dropout_p=p, seed=seed,
                                    offset=offset)
    fa.fa_device_status()
    return tuple(x.cpu() for x in (o, lse, dq, dk, dv))


def _oracle_varlen(q, k, v, do, cu_q, cu_k, causal, p=0.0, seed=0, offset=0):
    qf, kf, vf, dof = as_float64(q, k, v, do)
    cq, ck = cu_q.numpy(), cu_k.numpy()
    s = 1.0 / math.sqrt(q.shape[-1])
    if p == 0.0:
        o, lse = VL.forward_varlen(qf, kf, vf, cq, ck, s, causal)
        return (o, lse) + VL.backward_varlen(qf, kf, vf, dof, cq, ck, s, causal)
    # dropout: the keep mask of sequence b, head h is drawn with bh = b * H + h
    # and query / key indices counted within the sequence
    H = q.shape[1]
    c = DR.keep_scale(p)
    o, lse = np.zeros(qf.shape), np.full(qf.shape[:2], -np.inf)
    dq, dk, dv = np.zeros(qf.shape), np.zeros(kf.shape), np.zeros(vf.shape)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        for h in range(H):
            keep = DR.keep_mask(seed, offset, p, b * H + h, q1 - q0, k1 - k0)
            args = (qf[q0:q1, h], kf[k0:k1, h], vf[k0:k1, h])
            o[q0:q1, h], lse[q0:q1, h] = A.forward_head(*args, s, causal, keep=keep, keep_scale=c)
            dq[q0:q1, h], dk[k0:k1, h], dv[k0:k1, h] = A.backward_head(*args, dof[q0:q1, h], s, causal, keep=keep,
                                                                       keep_scale=c)
    return o, lse, dq, dk, dv


def _compare(got, want, dtype, o_tol=None):
    o, lse, dq, dk, dv = got
    ro, rl, rdq, rdk, rdv = want
    eo = float(np.abs(o.double().numpy() - ro).max())
    assert eo <= (o_tol or O_TOL[dtype]), eo
    gl = lse.double().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(rl))
    fin = np.isfinite(rl)
    if fin.any():
        assert float(np.abs(gl[fin] - rl[fin]).max()) <= LSE_TOL
    for n, g, r in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
        g = g.double().numpy()
        if np.linalg.norm(r) < 1e-12:
            assert np.abs(g).max() <= 1e-4, n
        else:
            e = rel_fro(g, r)
            assert e <= GRAD_REL_FRO, (n, e)


LENGTHS = [  # (query lengths, key lengths)
    ([300, 17, 129, 1], [300, 17, 129, 1]),
    ([64, 500, 3], [200, 513, 260]),       # Nq <= Nk: bottom-right diagonals off the tile grid
    ([260, 40, 130], [100, 40, 7]),        # Nq > Nk: rows that see no key under the causal mask
    ([0, 200, 5, 0], [50, 0, 77, 3]),      # empty query ranges and a sequence without keys
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lq,lk", LENGTHS)
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16"), (96, "bf16")])
def test_varlen_matches_oracle(causal, lq, lk, d, dtype):
    H = 2
    q, k, v, do, cu_q, cu_k = varlen_inputs(lq, lk, H, d, dtype, seed=sum(lq) + 3 * sum(lk) + d)
    got = _run_varlen(q, k, v, do, cu_q, cu_k, lq, lk, causal)
    _compare(got, _oracle_varlen(q, k, v, do, cu_q, cu_k, causal), dtype)


def test_varlen_with_dropout_matches_oracle():
    lq, lk = [200, 33, 300], [250, 33, 290]
    q, k, v, do, cu_q, cu_k = varlen_inputs(lq, lk, 2, 128, "bf16", seed=11)
    got = _run_varlen(q, k, v, do, cu_q, cu_k, lq, lk, True, p=0.2, seed=77, offset=4)
    want = _oracle_varlen(q, k, v, do, cu_q, cu_k, True, p=0.2, seed=77, offset=4)
    _compare(got, want, "bf16", o_tol=max(O_TOL["bf16"], 2.0 ** -8 * float(np.abs(want[0]).max())))


def test_one_sequence_equals_dense():
    """A batch of one sequence gives the dense kernels' O, LSE, dQ, dK, dV bit for bit."""
    N, H, d = 700, 3, 128
    q, k, v, do = attention_inputs(1, H, N, d, "bf16", seed=21)
    dense = [x.to(DEV) for x in (q, k, v, do)]
    o1, l1 = fa.forward(*dense[:3], causal=True)
    g1 = fa.backward(*dense[:3], o1, l1, dense[3], causal=True)
    packed = [x[0].transpose(0, 1).contiguous().to(DEV) for x in (q, k, v, do)]  # [N, H, d]
    cu = torch.tensor([0, N], dtype=torch.int32, device=DEV)
    o2, l2 = fa.forward_varlen(*packed[:3], cu, cu, N, N, causal=True)
    g2 = fa.backward_varlen(*packed[:3], o2, l2, packed[3], cu, cu, N, N, causal=True)
    fa.fa_device_status()
    t = lambda x: x.transpose(0, 1).unsqueeze(0)  # noqa: E731  [N, H, d] -> [1, H, N, d]
    assert torch.equal(o1, t(o2)) and torch.equal(l1, l2.T.unsqueeze(0))
    # both take the split backward (dQ by its own kernel, no atomics)
    assert torch.equal(g1[1], t(g2[1])) and torch.equal(g1[2], t(g2[2])) and torch.equal(g1[0], t(g2[0]))


def test_bad_offsets_are_reported_not_followed():
    """Offsets beyond the packed totals: the sequence is skipped and
    FA_ERR_SEQLENS is reported; the other sequences are still computed."""
    lq = [100, 50]
    q, k, v, do, cu_q, cu_k = varlen_inputs(lq, lq, 2, 64, "fp16", seed=5)
    bad_q = cu_q.clone()
    bad_q[2] = 1000  # beyond total_q = 150
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    o = torch.zeros_like(qd)
    lse = torch.zeros(qd.shape[:2], device=DEV)
    fa.fa_forward_varlen(qd, kd, vd, o, lse, bad_q.to(DEV), cu_k.to(DEV), 100, 100)
    with pytest.raises(fa.FAError) as e:
        fa.fa_device_status()
    assert e.value.code == 7
    want, _ = VL.forward_varlen(*as_float64(q, k, v), cu_q.numpy(), cu_k.numpy(), 1 / 8.0)
    assert float(np.abs(o[:100].double().cpu().numpy() - want[:100]).max()) <= O_TOL["fp16"]
    assert torch.all(o[100:] == 0)
    fa.fa_device_status()  # cleared


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,dtype", [(300, "bf16"), (777, "fp16")])
def test_head_dim_96_dense(causal, N, dtype):
    B, H, d = 1, 3, 96
    q, k, v, do = attention_inputs(B, H, N, d, dtype, seed=N + 96)
    dense = [x.to(DEV) for x in (q, k, v, do)]
    o, lse = fa.forward(*dense[:3], causal=causal)
    dq, dk, dv = fa.backward(*dense[:3], o, lse, dense[3], causal=causal)
    fa.fa_device_status()
    qf, kf, vf, dof = as_float64(q, k, v, do)
    s = 1 / math.sqrt(d)
    for h in range(H):
        ro, rl = A.forward_head(qf[0, h], kf[0, h], vf[0, h], s, causal)
        assert float(np.abs(o[0, h].double().cpu().numpy() - ro).max()) <= O_TOL[dtype]
        assert float(np.abs(lse[0, h].double().cpu().numpy() - rl).max()) <= LSE_TOL
        for g, r in zip((dq, dk, dv), A.backward_head(qf[0, h], kf[0, h], vf[0, h], dof[0, h], s, causal)):
            assert rel_fro(g[0, h].double().cpu().numpy(), r) <= GRAD_REL_FRO


def test_varlen_stages_equal_the_full_call():
    """fa_backward_varlen takes the split backward: preprocess on the flat
    [total_q * H, d] rows without an accumulator plus fa_backward_dk_dv_varlen
    and fa_backward_dq_varlen (the launches the benchmark times one by one)
    give its result bit for bit, and the accumulator region of its workspace
    stays untouched.  The accumulated stages (fa_backward_dkdv_varlen +
    dq_convert) agree."""
    lq = [300, 129, 700]
    q, k, v, do, cu_q, cu_k = (x.to(DEV) for x in varlen_inputs(lq, lq, 2, 128, "bf16", seed=31))
    L = max(lq)
    o, lse = fa.forward_varlen(q, k, v, cu_q, cu_k, L, L, causal=True)
    T, H, d = q.shape
    rows = T * H
    ws = torch.full((fa.fa_backward_varlen_workspace_size(T, H, d),), 0xA5, device=DEV, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_backward_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_q, cu_k, L, L, ws, causal=True)
    off = (rows * 4 + 255) // 256 * 256
    assert bool((ws[off:] == 0xA5).all())
    flat = lambda x: x.view(1, 1, rows, -1)  # noqa: E731
    delta = torch.empty((T, H), device=DEV, dtype=torch.float32)
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_backward_preprocess(flat(o), flat(do), delta.view(1, 1, rows), None)
    fa.fa_backward_dk_dv_varlen(q, k, v, do, lse, delta, dk2, dv2, cu_q, cu_k, L, L, causal=True)
    fa.fa_backward_dq_varlen(q, k, v, do, lse, delta, dq2, cu_q, cu_k, L, L, causal=True)
    fa.fa_device_status()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2) and torch.equal(dq, dq2)
    acc = torch.empty((T, H, d), device=DEV, dtype=torch.float32)
    dq3, dk3, dv3 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.fa_backward_preprocess(flat(o), flat(do), delta.view(1, 1, rows), flat(acc))
    fa.fa_backward_dkdv_varlen(q, k, v, do, lse, delta, acc, dk3, dv3, cu_q, cu_k, L, L, causal=True)
    fa.fa_backward_dq_convert(flat(acc), flat(dq3), scale=1 / math.sqrt(d))
    fa.fa_device_status()
    for x, y in ((dq, dq3), (dk, dk3), (dv, dv3)):
        assert float((x.float() - y.float()).abs().max()) <= 1e-2 * float(x.float().abs().max())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lq,lk", LENGTHS[1:])
def test_varlen_split_stages_match_oracle(causal, lq, lk):
    """The split stages alone against the oracle on rectangular sequences
    (bottom-right diagonals off the tile grid, rows that see no key, empty
    ranges)."""
    H, d = 2, 64
    q, k, v, do, cu_q, cu_k = varlen_inputs(lq, lk, H, d, "fp16", seed=7 + sum(lq) + sum(lk))
    qd, kd, vd, dod, cqd, ckd = (x.to(DEV) for x in (q, k, v, do, cu_q, cu_k))
    mq, mk = max(max(lq), 1), max(max(lk), 1)
    o, lse = fa.forward_varlen(qd, kd, vd, cqd, ckd, mq, mk, causal=causal)
    T = qd.shape[0]
    rows = T * H
    delta = torch.empty((T, H), device=DEV, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    fa.fa_backward_preprocess(o.view(1, 1, rows, -1), dod.view(1, 1, rows, -1), delta.view(1, 1, rows), None)
    fa.fa_backward_dk_dv_varlen(qd, kd, vd, dod, lse, delta, dk, dv, cqd, ckd, mq, mk, causal=causal)
    fa.fa_backward_dq_varlen(qd, kd, vd, dod, lse, delta, dq, cqd, ckd, mq, mk, causal=causal)
    fa.fa_device_status()
    got = tuple(x.cpu() for x in (o, lse, dq, dk, dv))
    _compare(got, _oracle_varlen(q, k, v, do, cu_q, cu_k, causal), "fp16")

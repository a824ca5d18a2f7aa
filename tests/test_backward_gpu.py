"""Backward parity: dQ, dK, dV from the CUDA path (through the C ABI) vs the
float64 oracle's explicit softmax backward, relative Frobenius error <= 1e-2.

Small and ragged sizes are compared on every head; the full-size workloads
on sampled heads (and, for the long ones, sampled query rows / key rows).
"""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_forward_gb300.synth import WORKLOADS, as_float64, attention_inputs, workload_inputs
from oracle import attention as A

from gpu_util import GRAD_REL_FRO, LSE_TOL, O_TOL, check_forward_heads, gpu_forward_backward, rel_fro

pytestmark = pytest.mark.gpu


def _check_grads(q, k, v, do, dq, dk, dv, causal, heads=None, rows=None, cols=None, scale=None):
    B, H, N, d = q.shape
    s = 1.0 / math.sqrt(d) if scale is None else scale
    qf, kf, vf, dof = as_float64(q, k, v, do)
    g = [x.to(torch.float64).numpy() for x in (dq, dk, dv)]
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    got = {n: [] for n in ("dq", "dk", "dv")}
    ref = {n: [] for n in ("dq", "dk", "dv")}
    for b, h in heads:
        if rows is None:
            rq, rk, rv = A.backward_head(qf[b, h], kf[b, h], vf[b, h], dof[b, h], s, causal)
            rr, cc = slice(None), slice(None)
        else:
            rq, rk, rv = A.backward_head_sampled(qf[b, h], kf[b, h], vf[b, h], dof[b, h], s, causal, rows, cols)
            rr, cc = rows, cols
        for n, x, r, idx in (("dq", g[0], rq, rr), ("dk", g[1], rk, cc), ("dv", g[2], rv, cc)):
            got[n].append(x[b, h][idx])
            ref[n].append(r)
    errs = {}
    for n in got:
        gn, rn = np.concatenate(got[n]), np.concatenate(ref[n])
        if np.linalg.norm(rn) == 0.0:
            # A single visible key makes dS = 0 exactly (P = 1): dQ = dK = 0,
            # so only an absolute bound on the rounding noise is meaningful.
            errs[n] = float(np.abs(gn).max())
            assert errs[n] <= 1e-4, (n, errs)
        else:
            errs[n] = rel_fro(gn, rn)
            assert np.isfinite(errs[n]) and errs[n] <= GRAD_REL_FRO, (n, errs)
    return errs


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 3, 64, 65, 127, 128, 129, 200, 383])
def test_backward_small_ragged(N, causal, d, dtype):
    q, k, v, do = attention_inputs(1, 2, N, d, dtype, seed=2000 + N + d)
    o, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, causal)
    eo, el = check_forward_heads(q, k, v, o, lse, causal)
    assert eo <= O_TOL[dtype] and el <= LSE_TOL, (eo, el)
    _check_grads(q, k, v, do, dq, dk, dv, causal)


def test_backward_scale():
    q, k, v, do = attention_inputs(2, 2, 300, 128, "bf16", seed=31, k_row_scale=True)
    o, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, True, scale=0.3)
    _check_grads(q, k, v, do, dq, dk, dv, True, scale=0.3)


def test_backward_c2_all_heads():
    """Workload C2: B=4, H=16, N=1024, d=64, fp16, causal -- every head."""
    w = WORKLOADS["C2"]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, w.causal)
    eo, el = check_forward_heads(q, k, v, o, lse, w.causal)
    assert eo <= O_TOL[w.dtype] and el <= LSE_TOL, (eo, el)
    _check_grads(q, k, v, do, dq, dk, dv, w.causal)


@pytest.mark.parametrize("name", ["C3N", "C3C"])
def test_backward_c3_sampled_heads(name):
    w = WORKLOADS[name]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, w.causal)
    heads = [(0, 0), (1, 15)]
    eo, el = check_forward_heads(q, k, v, o, lse, w.causal, heads=heads)
    assert eo <= O_TOL[w.dtype] and el <= LSE_TOL, (eo, el)
    _check_grads(q, k, v, do, dq, dk, dv, w.causal, heads=heads)


@pytest.mark.parametrize("name", ["C4", "C5"])
def test_backward_full_size_sampled(name):
    w = WORKLOADS[name]
    q, k, v, do = workload_inputs(w)
    o, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, w.causal)
    rng = np.random.default_rng(1)
    pick = np.unique(np.concatenate([[0, 1, 127, 128, w.N // 2, w.N - 1], rng.integers(0, w.N, 42)]))
    heads = [(w.B - 1, w.H - 1)] if name == "C5" else [(0, 0), (w.B - 1, w.H - 1)]
    eo, el = check_forward_heads(q, k, v, o, lse, w.causal, heads=heads, rows=pick)
    assert eo <= O_TOL[w.dtype] and el <= LSE_TOL, (eo, el)
    _check_grads(q, k, v, do, dq, dk, dv, w.causal, heads=heads, rows=pick, cols=pick)
    # dQ on every head (every L2 head group of every kernel), on a few rows each
    qf, kf, vf, dof = as_float64(q, k, v, do)
    s = 1.0 / math.sqrt(w.d)
    for b in range(w.B):
        for h in range(w.H):
            few = np.unique(np.concatenate([[0, 127, 128, w.N - 1], rng.integers(0, w.N, 4)]))
            ref = A.backward_head_rows(qf[b, h], kf[b, h], vf[b, h], dof[b, h], s, w.causal, few)
            err = rel_fro(dq[b, h].double().numpy()[few], ref)
            assert err <= GRAD_REL_FRO, (b, h, err)
    # Invariants that hold at any size (P rows sum to 1): sum_j dK_j = 0 and
    # sum_j dV_j = sum_i dO_i, per head, up to the rounding of the inputs.
    dkf = dk.float().sum(dim=2)
    assert float(dkf.abs().max()) <= 1e-2 * float(dk.float().abs().sum(dim=2).max())
    dvs, dos = dv.float().sum(dim=2), do.float().sum(dim=2)
    assert float((dvs - dos).abs().max()) <= 1e-2 * float(dos.abs().max() + 1)


def test_backward_several_head_groups_with_a_partial_last_one():
    """B*H = 40 heads at N = 4096, d = 128: the forward and dQ kernels take
    heads in L2 groups of 32, the dK/dV kernels in groups of 16, so both see
    full groups and a partial last group.  Every head is compared on sampled
    rows (O, LSE, dQ); dK and dV on sampled keys of heads in the first, a
    middle and the partial last group."""
    B, H, N, d = 5, 8, 4096, 128
    q, k, v, do = attention_inputs(B, H, N, d, "bf16", seed=4040)
    o, lse, dq, dk, dv = gpu_forward_backward(q, k, v, do, True)
    rng = np.random.default_rng(40)
    qf, kf, vf, dof = as_float64(q, k, v, do)
    s = 1.0 / math.sqrt(d)
    for b in range(B):
        for h in range(H):
            few = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 4)]))
            eo, el = check_forward_heads(q, k, v, o, lse, True, heads=[(b, h)], rows=few)
            assert eo <= O_TOL["bf16"] and el <= LSE_TOL, (b, h, eo, el)
            ref = A.backward_head_rows(qf[b, h], kf[b, h], vf[b, h], dof[b, h], s, True, few)
            err = rel_fro(dq[b, h].double().numpy()[few], ref)
            assert err <= GRAD_REL_FRO, (b, h, err)
    pick = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.integers(0, N, 27)]))
    heads = [(0, 0), (2, 1), (4, 7)]  # flat heads 0, 17 and 39
    _check_grads(q, k, v, do, dq, dk, dv, True, heads=heads, rows=pick, cols=pick)

"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI binding and compare with the float64 oracle on the same inputs."""
import math

import numpy as np
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import as_float64
from oracle import attention as A

# Tolerances fixed by the specification of the path.
O_TOL = {"fp16": 2e-3, "bf16": 1e-2}    # forward O, max abs
LSE_TOL = 1e-3                          # forward LSE, max abs (both dtypes)
GRAD_REL_FRO = 1e-2                     # dQ, dK, dV relative Frobenius


def dtype_name(t):
    return "bf16" if t.dtype == torch.bfloat16 else "fp16"


def gpu_forward(q, k, v, causal, scale=None):
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    fa.fa_device_status()
    return o.cpu(), lse.cpu()


def gpu_forward_backward(q, k, v, do, causal, scale=None):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    fa.fa_device_status()
    return tuple(x.cpu() for x in (o, lse, dq, dk, dv))


def check_forward_heads(q, k, v, o, lse, causal, heads=None, scale=None, rows=None):
    """Compare O and LSE with the oracle on selected (b, h) heads (all by default)
    and selected query rows (all by default).  Returns (max O err, max LSE err)."""
    B, H, N, d = q.shape
    s = 1.0 / math.sqrt(d) if scale is None else scale
    qf, kf, vf = as_float64(q, k, v)
    of = o.to(torch.float64).numpy()
    lf = lse.to(torch.float64).numpy()
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    eo = el = 0.0
    for b, h in heads:
        r = np.arange(N) if rows is None else np.asarray(rows)
        ro, rl = A.forward_head(qf[b, h], kf[b, h], vf[b, h], s, causal, rows=r)
        eo = max(eo, float(np.abs(of[b, h][r] - ro).max()))
        el = max(el, float(np.abs(lf[b, h][r] - rl).max()))
    assert np.isfinite(of).all() and np.isfinite(lf).all()
    return eo, el


def rel_fro(got, want):
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))

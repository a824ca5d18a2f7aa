"""The largest problem the interface accepts (B*H*N*d just below 2^31 elements,
N = 2^20 - 1 keys per head): causal forward on sampled rows against the
float64 oracle, so that no index arithmetic overflows at the size limit."""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import device_inputs
from oracle import attention as A

from gpu_util import LSE_TOL, O_TOL

pytestmark = pytest.mark.gpu


def test_forward_at_the_size_limit():
    B, H, N, d = 1, 16, (1 << 20) - 1, 128
    assert B * H * N * d < (1 << 31)
    dev = torch.device("cuda:0")
    q, k, v = device_inputs(B, H, N, d, "bf16", seed=99, device=dev)
    o, lse = fa.forward(q, k, v, causal=True)
    fa.fa_device_status()
    rows = np.array([0, 1, 127, 128, 255, 4097, N // 2, N - 129, N - 2, N - 1])
    s = 1.0 / math.sqrt(d)
    for h in (0, H - 1):
        qf, kf, vf = (x[0, h].double().cpu().numpy() for x in (q, k, v))
        ro, rl = A.forward_head(qf, kf, vf, s, True, rows=rows)
        eo = float(np.abs(o[0, h, rows].double().cpu().numpy() - ro).max())
        el = float(np.abs(lse[0, h, rows].double().cpu().numpy() - rl).max())
        assert eo <= O_TOL["bf16"] and el <= LSE_TOL, (h, eo, el)

"""fa_backward_noalloc: the backward pass for callers that cannot allocate
device memory (plugins whose host framework owns every allocation,
allocation-free serving paths, code that only receives raw pointers).

It must give the same dQ, dK, dV as fa_backward (which takes a caller
workspace), call after call, although every call reuses the same fixed
device scratch array.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300 import _lib
from exact_io_aware_forward_gb300.synth import attention_inputs

from gpu_util import GRAD_REL_FRO, rel_fro

SCRATCH_BYTES = 32 << 20


def test_rejects_problems_beyond_the_scratch():
    """Workspace above 32 MiB -> FA_ERR_SCRATCH_TOO_SMALL before any launch."""
    from exact_io_aware_forward_gb300 import build as fa_build
    fa_build.build()
    lib = _lib.lib()
    B, H, N, d = 1, 64, 2048, 128
    assert lib.fa_backward_workspace_size(B, H, N, d) > SCRATCH_BYTES
    ptr = 1 << 20  # never dereferenced: the size check comes first
    rc = lib.fa_backward_noalloc(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, B, H, N, d, 1, 1, 0.1, None)
    assert rc == 6
    assert "32 MiB" in _lib.status_string(rc)


BAD_CALLS = {
    # name: (argument overrides); every pointer is aligned and never dereferenced
    "zero_batch_d96": dict(B=0, d=96),
    "zero_n_d256": dict(N=0, d=256),
    "beyond_2_31": dict(H=16, N=1 << 20, d=128),
    "head_dim_80": dict(d=80),
    "dtype_7": dict(dt=7),
    "nan_scale": dict(scale=float("nan")),
    "negative_scale": dict(scale=-0.5),
    "null_q": dict(q=None),
    "null_lse": dict(lse=None),
    "misaligned_dq": dict(dq=(1 << 20) + 4),
    "misaligned_dv": dict(dv=(1 << 20) + 8),
}


@pytest.mark.parametrize("case", sorted(BAD_CALLS))
def test_invalid_arguments_get_the_status_of_fa_backward(case):
    """Both entry points reject the same bad call with the same status, before
    any launch (the pointers are never dereferenced; no GPU is needed)."""
    from exact_io_aware_forward_gb300 import build as fa_build
    fa_build.build()
    lib = _lib.lib()
    ptr = 1 << 20
    a = dict(q=ptr, k=ptr, v=ptr, o=ptr, do=ptr, lse=ptr, dq=ptr, dk=ptr, dv=ptr, B=1, H=2, N=64, d=64, dt=1,
             causal=1, scale=0.125)
    a.update(BAD_CALLS[case])
    tensors = [a[n] for n in ("q", "k", "v", "o", "do", "lse", "dq", "dk", "dv")]
    rest = [a["B"], a["H"], a["N"], a["d"], a["dt"], a["causal"], a["scale"]]
    want = lib.fa_backward(*tensors, *rest, ptr, 1 << 30, None)
    got = lib.fa_backward_noalloc(*tensors, *rest, None)
    assert want in (1, 2), _lib.status_string(want)
    assert got == want, (_lib.status_string(got), _lib.status_string(want))


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,dtype,causal", [(1, 4, 1000, 128, "bf16", True),
                                                   (2, 3, 515, 64, "fp16", False),
                                                   (1, 2, 600, 96, "bf16", True),
                                                   (1, 2, 400, 256, "bf16", True)])
def test_noalloc_matches_workspace_backward(B, H, N, d, dtype, causal):
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in attention_inputs(B, H, N, d, dtype, seed=4242 + N))
    o, lse = fa.forward(q, k, v, causal=causal)
    ref = fa.backward(q, k, v, o, lse, do, causal=causal)
    fa.fa_device_status()
    for call in range(2):  # the scratch keeps the previous call's contents
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        fa.fa_backward_noalloc(q, k, v, o, do, lse, dq, dk, dv, causal=causal)
        fa.fa_device_status()
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            g = got.double().cpu().numpy()
            r = want.double().cpu().numpy()
            err = rel_fro(g, r)
            assert err <= GRAD_REL_FRO, (call, name, err)

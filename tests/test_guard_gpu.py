"""No write outside the outputs: every output (and workspace) a call receives
is carved out of a larger buffer whose bytes before and after it hold a
sentinel pattern; after the call the sentinel must be intact.  This stands in
for a memory checker: the parity tests cannot see a write past the end of O,
LSE, dQ, dK, dV, which is the risk at ragged N, in packed tails, at d = 96
(the kernels compute with 128 features) and in the TMA-stored epilogues.

Sizes: ragged N (1, 129, 383), several heads, both strategies of the backward
(split: dense d <= 128; accumulated: dropout, block mask, d = 256), packed
variable-length batches with tails, split-KV decoding.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import attention_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GUARD = 4096  # bytes on each side (a multiple of 16: the carved tensor stays 16-byte aligned)
SENTINEL = 0xA7


class Guarded:
    """A tensor of `shape`/`dtype` inside a byte buffer with GUARD sentinel bytes on each side."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.buf = torch.full((n + 2 * GUARD,), SENTINEL, device=DEV, dtype=torch.uint8)
        self.n = n
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(*shape)

    def intact(self):
        head, tail = self.buf[:GUARD], self.buf[GUARD + self.n:]
        return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


def _check(*gs):
    torch.cuda.synchronize()
    fa.fa_device_status()
    for name, g in gs:
        assert g.intact(), name


@pytest.mark.parametrize("d", [64, 96, 128, 256])
@pytest.mark.parametrize("N", [1, 129, 383])
def test_dense_forward_and_backward_stay_inside_their_outputs(N, d):
    B, H = 2, 3
    q, k, v, do = (x.to(DEV) for x in attention_inputs(B, H, N, d, "bf16", seed=900 + N + d))
    go, gl = Guarded(q.shape, q.dtype), Guarded((B, H, N), torch.float32)
    fa.fa_forward(q, k, v, go.t, gl.t, True)
    _check(("o", go), ("lse", gl))
    gq, gk, gv = (Guarded(q.shape, q.dtype) for _ in range(3))
    gw = Guarded((fa.fa_backward_workspace_size(B, H, N, d),), torch.uint8)
    fa.fa_backward(q, k, v, go.t, do, gl.t, gq.t, gk.t, gv.t, gw.t, True)
    _check(("dq", gq), ("dk", gk), ("dv", gv), ("workspace", gw))
    assert torch.isfinite(gq.t.float()).all() and torch.isfinite(gk.t.float()).all()


@pytest.mark.parametrize("d", [96, 128])
def test_accumulated_backward_paths_stay_inside_their_outputs(d):
    """Dropout and block-mask calls take the accumulated strategy (fp32 dQ
    reductions into the workspace, then the convert kernel)."""
    B, H, N = 1, 2, 383
    q, k, v, do = (x.to(DEV) for x in attention_inputs(B, H, N, d, "bf16", seed=950 + d))
    T = (N + 127) // 128
    mask = torch.ones((1, T, T), device=DEV, dtype=torch.uint8)
    mask[0, 2, 0] = 0
    for kw in ({"dropout_p": 0.1, "seed": 5, "offset": 3}, {"block_mask": mask}):
        go, gl = Guarded(q.shape, q.dtype), Guarded((B, H, N), torch.float32)
        if "block_mask" in kw:
            fa.fa_forward_blocksparse(q, k, v, go.t, gl.t, mask, True)
        else:
            fa.fa_forward_dropout(q, k, v, go.t, gl.t, 0.1, 5, 3, True)
        _check(("o", go), ("lse", gl))
        gq, gk, gv = (Guarded(q.shape, q.dtype) for _ in range(3))
        gw = Guarded((fa.fa_backward_workspace_size(B, H, N, d),), torch.uint8)
        if "block_mask" in kw:
            fa.fa_backward_blocksparse(q, k, v, go.t, do, gl.t, gq.t, gk.t, gv.t, mask, gw.t, True)
        else:
            fa.fa_backward_dropout(q, k, v, go.t, do, gl.t, gq.t, gk.t, gv.t, gw.t, 0.1, 5, 3, True)
        _check(("dq", gq), ("dk", gk), ("dv", gv), ("workspace", gw))


@pytest.mark.parametrize("d", [96, 128])
def test_packed_batches_stay_inside_their_outputs(d):
    lens = [1, 130, 383, 77]
    H = 3
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=DEV)
    T = int(sum(lens))
    q, k, v, do = (x.to(DEV)[0].permute(1, 0, 2).contiguous()
                   for x in attention_inputs(1, H, T, d, "bf16", seed=960 + d))  # [T, H, d]
    L = max(lens)
    go, gl = Guarded(q.shape, q.dtype), Guarded((T, H), torch.float32)
    fa.fa_forward_varlen(q, k, v, go.t, gl.t, cu, cu, L, L, True)
    _check(("o", go), ("lse", gl))
    gq, gk, gv = (Guarded(q.shape, q.dtype) for _ in range(3))
    gw = Guarded((fa.fa_backward_varlen_workspace_size(T, H, d),), torch.uint8)
    fa.fa_backward_varlen(q, k, v, go.t, do, gl.t, gq.t, gk.t, gv.t, cu, cu, L, L, gw.t, True)
    _check(("dq", gq), ("dk", gk), ("dv", gv), ("workspace", gw))


@pytest.mark.parametrize("Nq,Nk,d", [(1, 1000, 128), (5, 4097, 64), (16, 300, 256)])
def test_decoding_stays_inside_its_outputs(Nq, Nk, d):
    B, H = 2, 3
    q = attention_inputs(B, H, Nq, d, "bf16", seed=970, with_do=False)[0].to(DEV)
    _, k, v, _ = attention_inputs(B, H, Nk, d, "bf16", seed=971, with_do=False)
    k, v = k.to(DEV), v.to(DEV)
    go, gl = Guarded(q.shape, q.dtype), Guarded((B, H, Nq), torch.float32)
    gw = Guarded((fa.fa_decode_workspace_size(B, H, Nq, Nk, d, 0),), torch.uint8)
    fa.fa_forward_decode(q, k, v, go.t, gl.t, gw.t, True)
    _check(("o", go), ("lse", gl), ("workspace", gw))

"""Peak device memory of a forward + backward through the public API grows
linearly in N (nothing N x N is ever allocated): measured with torch's
allocator statistics at N and 2N, inputs included."""
import pytest
import torch

import exact_io_aware_forward_gb300 as fa

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _peak(N, B=1, H=8, d=128):
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(DEV)
    torch.cuda.reset_peak_memory_stats(DEV)
    g = torch.Generator(device="cuda").manual_seed(N)
    q, k, v, do = (torch.randn(B, H, N, d, device=DEV, dtype=torch.bfloat16, generator=g) for _ in range(4))
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True)
    fa.fa_device_status()
    peak = torch.cuda.max_memory_allocated(DEV) - base
    del q, k, v, do, o, lse, dq, dk, dv
    return peak


def test_peak_memory_is_linear_in_n():
    p1, p2 = _peak(8192), _peak(16384)
    assert p2 <= 2.05 * p1, (p1, p2)
    # what the naive S and P alone would need at 16384 (2 x N^2 x 2 bytes per head, 8 heads)
    naive = 2 * 16384 * 16384 * 2 * 8
    assert p2 < naive / 10, (p2, naive)
    # and the peak is the tensors themselves: 9 16-bit [N, d] arrays per head (q, k, v, dO, O,
    # dQ, dK, dV) plus LSE and the workspace (D and the float32 dQ accumulator)
    per_head = 16384 * 128 * 2 * 8 + 16384 * 4 + 16384 * (4 + 4 * 128)
    assert p2 <= 8 * per_head * 1.05 + (64 << 20), (p2, 8 * per_head)

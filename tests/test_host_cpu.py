"""Host-side logic on the CPU: the workload recipes (shapes, seeds, the
K-row scaling of C3, block masks, packed lengths) and the work counts the
benchmark divides by, each against an independent closed form."""
import math
import os
import sys

import numpy as np
import pytest
import torch

from exact_io_aware_forward_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


# (B, H, N, d, dtype, causal, forward FLOP) of the five specified workloads;
# the FLOP column is 4 B H N^2 d, halved under the causal mask, as printed in
# the workload table (16.8 MFLOP, 8.59 GFLOP, 137.4 / 68.7 GFLOP, 1099.5 GFLOP,
# 2199.0 GFLOP).
TABLE = {
    "C1": (1, 1, 256, 64, "fp16", False, 16.8e6),
    "C2": (4, 16, 1024, 64, "fp16", True, 8.59e9),
    "C3N": (2, 16, 4096, 64, "bf16", False, 137.4e9),
    "C3C": (2, 16, 4096, 64, "bf16", True, 68.7e9),
    "C4": (2, 32, 8192, 128, "bf16", True, 1099.5e9),
    "C5": (1, 8, 32768, 128, "bf16", True, 2199.0e9),
}


@pytest.mark.parametrize("name", sorted(TABLE))
def test_workloads_match_the_table(name):
    B, H, N, d, dtype, causal, flops = TABLE[name]
    w = synth.WORKLOADS[name]
    assert (w.B, w.H, w.N, w.d, w.dtype, w.causal) == (B, H, N, d, dtype, causal)
    assert abs(w.fwd_flops() - flops) <= 0.005 * flops
    assert w.k_row_scale == name.startswith("C3")


def test_inputs_are_seeded_16_bit_normals():
    a = synth.attention_inputs(1, 2, 300, 64, "bf16", seed=5)
    b = synth.attention_inputs(1, 2, 300, 64, "bf16", seed=5)
    c = synth.attention_inputs(1, 2, 300, 64, "bf16", seed=6)
    for x, y, z in zip(a, b, c):
        assert x.dtype == torch.bfloat16 and x.shape == (1, 2, 300, 64)
        assert torch.equal(x, y) and not torch.equal(x, z)
        f = x.double()
        assert abs(float(f.mean())) < 0.03 and abs(float(f.std()) - 1.0) < 0.03
    q16 = synth.attention_inputs(1, 1, 64, 64, "fp16", seed=5, with_do=False)
    assert q16[0].dtype == torch.float16 and q16[3] is None


def test_k_rows_scaled_by_uniform_factors():
    """C3's recipe: each K row is multiplied by a factor from U(0.5, 3) drawn
    after Q, K, V; Q and V are the unscaled draws."""
    q0, k0, v0, _ = synth.attention_inputs(1, 2, 512, 64, "fp16", seed=9)
    q1, k1, v1, _ = synth.attention_inputs(1, 2, 512, 64, "fp16", seed=9, k_row_scale=True)
    assert torch.equal(q0, q1) and torch.equal(v0, v1)
    ratio = (k1.double().norm(dim=-1) / k0.double().norm(dim=-1)).flatten().numpy()
    assert ratio.min() >= 0.5 * (1 - 2e-3) and ratio.max() <= 3.0 * (1 + 2e-3)
    # uniform over [0.5, 3]: mean 1.75, standard deviation 2.5 / sqrt(12)
    assert abs(ratio.mean() - 1.75) < 6 * (2.5 / math.sqrt(12)) / math.sqrt(ratio.size)
    # the factor is per row: every element of a row is scaled alike
    per_elem = (k1.double() / k0.double().where(k0.double().abs() > 0.25, torch.tensor(float("nan"))))
    spread = np.nanmax(per_elem.numpy(), axis=-1) / np.nanmin(per_elem.numpy(), axis=-1)
    assert np.nanmax(spread) < 1.01


def test_block_mask_recipe():
    w = synth.S1
    bm = synth.block_mask(w)
    T = w.tiles
    assert bm.shape == (1, T, T) and bm.dtype == bool and T == 64
    assert bm[0, np.arange(T), np.arange(T)].all()
    off = ~np.eye(T, dtype=bool)
    frac = bm[0][off].mean()
    n = off.sum()
    assert abs(frac - w.density) < 6 * math.sqrt(w.density * (1 - w.density) / n)
    assert np.array_equal(bm, synth.block_mask(w))


@pytest.mark.parametrize("N", [256, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_flops_counts_pairs(N, causal):
    """All blocks kept: the dense pair count, N^2 or N(N+1)/2, times 4 d per
    pair and head; one block kept: its own pairs (ragged sizes included)."""
    w = synth.BlockSparseWorkload("t", 2, 3, N, 64, "bf16", causal, 1.0, False, 0)
    T = w.tiles
    ones = np.ones((1, T, T), bool)
    pairs = N * (N + 1) / 2 if causal else N * N
    assert bench.block_mask_flops(w, ones) == pytest.approx(4.0 * 64 * 6 * pairs)
    one = np.zeros((6, T, T), bool)  # per-head masks: only head 0 keeps block (T-1, 0)
    one[0, T - 1, 0] = True
    rows = N - 128 * (T - 1)
    assert bench.block_mask_flops(w, one) == pytest.approx(4.0 * 64 * rows * 128)


def test_varlen_recipe_and_pairs():
    w = synth.V1
    assert w.B == 16 and all(256 <= n <= 8192 for n in w.lengths)
    assert sum(w.lengths) == 66921
    assert bench.varlen_pairs(w.lengths, True) == sum(n * (n + 1) // 2 for n in w.lengths)
    assert bench.varlen_pairs([3, 5], False) == 9 + 25
    assert bench.variant_flops("varlen", w, None) == 4.0 * w.d * w.H * bench.varlen_pairs(w.lengths, True)
    q, k, v, do, cu_q, cu_k = synth.varlen_inputs([3, 0, 5], [4, 2, 5], 2, 64, "bf16", seed=1)
    assert q.shape == (8, 2, 64) and k.shape == (11, 2, 64) and do.shape == (8, 2, 64)
    assert cu_q.tolist() == [0, 3, 3, 8] and cu_k.tolist() == [0, 4, 6, 11]
    assert cu_q.dtype == torch.int32

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


def test_roofline_traffic_is_tied_to_the_captured_sources(tmp_path):
    """The bench reports a captured DRAM traffic only while the kernel's source
    files hash as they did at capture time."""
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    good = tmp_path / "good.md"
    good.write_text(f"x\ntraffic_bytes_per_launch: 1234\nsource_sha256_16: `{h}`\n")
    assert bench.captured_traffic(str(good))[0] == 1234
    stale = tmp_path / "stale.md"
    stale.write_text("traffic_bytes_per_launch: 1234\nsource_sha256_16: 0000000000000000\n")
    assert bench.captured_traffic(str(stale)) == (None, "kernel changed since the capture")
    assert bench.captured_traffic(str(tmp_path / "absent.md"))[0] is None


def test_dkdv_flop_factor_follows_the_backward_strategy():
    assert bench.dkdv_factor("dense", synth.C4) == 2.0
    assert bench.dkdv_factor("dense", synth.W256) == 2.5
    assert bench.dkdv_factor("dropout", synth.C4) == 2.5
    assert bench.dkdv_factor("blocksparse", synth.S1) == 2.0
    assert bench.dkdv_factor("varlen", synth.V1) == 2.0


def _exp2_poly_f32(x):
    """The kernels' FMA-pipe 2^x (exp2_poly2 in fa_ptx.cuh) step by step in
    float32: clamp, round by adding 1.5 * 2^23, cubic in f, exponent add."""
    f32 = np.float32
    x = np.maximum(x.astype(f32), f32(-125.0))
    t = (x + f32(12582912.0)).astype(f32)
    n = (t + f32(-12582912.0)).astype(f32)
    f = (n * f32(-1.0) + x).astype(f32)
    p = (f * f32(0.0551716685) + f32(0.242611140)).astype(f32)
    p = (p * f + f32(0.693260968)).astype(f32)
    p = (p * f + f32(0.999928057)).astype(f32)
    bits = p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_fma_pipe_exp2_error_bound():
    """Relative error below 1e-4 (under half an ulp of P rounded to fp16) over
    the range the softmax uses, exact powers of two at integers, and the
    clamp below -125."""
    x = np.concatenate([np.linspace(-125, 20, 400001), -np.logspace(-6, 2, 2001), np.arange(-120, 21)])
    got = _exp2_poly_f32(x).astype(np.float64)
    want = np.exp2(np.maximum(x, -125.0))
    rel = np.abs(got / want - 1)
    assert rel.max() < 1e-4, rel.max()
    ints = np.arange(-120, 21).astype(np.float64)
    assert np.abs(_exp2_poly_f32(ints) / np.exp2(ints) - 1).max() < 1e-4
    low = _exp2_poly_f32(np.array([-np.inf, -1e30, -200.0]))
    assert np.all(low > 0) and np.all(low < 3e-38)


def test_committed_dkdv_profiles_carry_traffic_and_hash():
    """Every profile the bench lines read records a traffic figure and a source hash."""
    import re
    for path in (bench.DKDV_PROFILE, *bench.VARIANT_PROFILES.values()):
        text = open(path, encoding="utf-8").read()
        assert re.search(r"^traffic_bytes_per_launch: \d+$", text, re.M), path
        assert re.search(r"^source_sha256_16: `[0-9a-f]{16}`$", text, re.M), path

"""Forward parity: CUDA path (through the C ABI) vs the float64 oracle.

Small and ragged sizes are compared element by element on every head; the
full-size workloads are compared on sampled heads / rows in the same launch
configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

from exact_io_aware_forward_gb300.synth import WORKLOADS, attention_inputs, workload_inputs

from gpu_util import LSE_TOL, O_TOL, check_forward_heads, dtype_name, gpu_forward

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 3, 127, 128, 129, 200, 256, 383, 640])
def test_forward_small_ragged(N, causal, d, dtype):
    q, k, v, _ = attention_inputs(1, 2, N, d, dtype, seed=1000 + N + d, with_do=False)
    o, lse = gpu_forward(q, k, v, causal)
    eo, el = check_forward_heads(q, k, v, o, lse, causal)
    assert eo <= O_TOL[dtype], eo
    assert el <= LSE_TOL, el


@pytest.mark.parametrize("scale", [0.05, 0.5, 1.0])
def test_forward_scale_and_wide_scores(scale):
    """Caller-chosen scale; scores spanning tens of units exercise the rescale.

    Outside the specified workloads a near-one-hot softmax makes |O| approach
    max|V|; P rounded to bf16 (relative 2^-9) and O rounded to bf16 (2^-9 of
    |O|) then bound the error by 2^-8 * max|V|, which can exceed the fixed
    1e-2.  The bound used is the larger of the two.
    """
    q, k, v, _ = attention_inputs(2, 3, 513, 64, "bf16", seed=77, k_row_scale=True, with_do=False)
    o, lse = gpu_forward(q, k, v, True, scale=scale)
    eo, el = check_forward_heads(q, k, v, o, lse, True, scale=scale)
    tol = max(O_TOL["bf16"], 2.0 ** -8 * float(v.float().abs().max()))
    assert eo <= tol and el <= LSE_TOL, (eo, el, tol)


def test_forward_c1():
    """Workload C1: B=1, H=1, N=256, d=64, fp16, non-causal -- every element."""
    w = WORKLOADS["C1"]
    q, k, v, _ = workload_inputs(w)
    o, lse = gpu_forward(q, k, v, w.causal)
    eo, el = check_forward_heads(q, k, v, o, lse, w.causal)
    assert eo <= O_TOL["fp16"], eo
    assert el <= LSE_TOL, el


def test_forward_c2_all_heads():
    w = WORKLOADS["C2"]
    q, k, v, _ = workload_inputs(w, with_do=False)
    o, lse = gpu_forward(q, k, v, w.causal)
    eo, el = check_forward_heads(q, k, v, o, lse, w.causal)
    assert eo <= O_TOL[w.dtype] and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("name", ["C3N", "C3C"])
def test_forward_c3_sampled_heads(name):
    w = WORKLOADS[name]
    q, k, v, _ = workload_inputs(w, with_do=False)
    o, lse = gpu_forward(q, k, v, w.causal)
    heads = [(0, 0), (1, 7), (1, 15)]
    eo, el = check_forward_heads(q, k, v, o, lse, w.causal, heads=heads)
    assert eo <= O_TOL[w.dtype] and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("name", ["C4", "C5"])
def test_forward_full_size_sampled_rows(name):
    """Every head of the full-size workloads (so every L2 head group and every
    position inside one), on the tile-edge rows and a few random rows; two
    heads on 64 rows."""
    w = WORKLOADS[name]
    q, k, v, _ = workload_inputs(w, with_do=False)
    o, lse = gpu_forward(q, k, v, w.causal)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, w.N - 1], rng.integers(0, w.N, 58)]))
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    eo, el = check_forward_heads(q, k, v, o, lse, w.causal, heads=heads, rows=rows)
    assert eo <= O_TOL[w.dtype] and el <= LSE_TOL, (eo, el)
    for b in range(w.B):
        for h in range(w.H):
            few = np.unique(np.concatenate([[0, 127, 128, w.N - 1], rng.integers(0, w.N, 4)]))
            eo, el = check_forward_heads(q, k, v, o, lse, w.causal, heads=[(b, h)], rows=few)
            assert eo <= O_TOL[w.dtype] and el <= LSE_TOL, (b, h, eo, el)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [2047, 2048, 2049, 3000])
def test_forward_d128_around_the_persistence_threshold(N, causal):
    """d = 128 dense attention is dispatched by key length and mask: causal
    runs persistent CTAs up to 2048 keys and one CTA per item above, non-causal
    runs the one-shot kernel.  Every head of B = 2, H = 5 (a partial L2 head
    group) on tile-edge and random rows."""
    B, H, d = 2, 5, 128
    q, k, v, _ = attention_inputs(B, H, N, d, "bf16", seed=900 + N + causal, with_do=False)
    o, lse = gpu_forward(q, k, v, causal)
    rng = np.random.default_rng(N)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, N - 2, N - 1], rng.integers(0, N, 24)]))
    eo, el = check_forward_heads(q, k, v, o, lse, causal, rows=rows)
    assert eo <= O_TOL["bf16"] and el <= LSE_TOL, (eo, el)

"""Split-KV decoding (few queries, many keys): CUDA path vs the float64 oracle.

The oracle evaluates each head without any split; the GPU result must agree
for every split count, including splits that see no visible key.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import as_float64, attention_inputs
from oracle import attention as A

from gpu_util import LSE_TOL, O_TOL

pytestmark = pytest.mark.gpu


def _inputs(B, H, Nq, Nk, d, dtype, seed):
    q, _, _, _ = attention_inputs(B, H, Nq, d, dtype, seed=seed, with_do=False)
    _, k, v, _ = attention_inputs(B, H, Nk, d, dtype, seed=seed + 1, with_do=False)
    return q, k, v


def _check(q, k, v, o, lse, causal, heads=None):
    B, H, Nq, d = q.shape
    s = 1.0 / math.sqrt(d)
    qf, kf, vf = as_float64(q, k, v)
    of, lf = o.double().numpy(), lse.double().numpy()
    eo = el = 0.0
    for b, h in heads or [(b, h) for b in range(B) for h in range(H)]:
        ro, rl = A.forward_head(qf[b, h], kf[b, h], vf[b, h], s, causal)
        eo = max(eo, float(np.abs(of[b, h] - ro).max()))
        el = max(el, float(np.abs(lf[b, h] - rl).max()))
    return eo, el


CASES = [
    (1, 2, 1, 1, 128, "bf16", False, 0), (1, 2, 1, 5, 64, "fp16", True, 0), (2, 3, 1, 300, 128, "bf16", True, 0),
    (1, 2, 3, 1000, 64, "bf16", True, 7), (1, 2, 4, 1000, 128, "fp16", False, 3), (2, 2, 5, 4100, 128, "bf16", True, 0),
    (1, 3, 16, 700, 64, "fp16", True, 1), (1, 2, 17, 2000, 128, "bf16", True, 9), (1, 1, 40, 40, 128, "bf16", True, 0),
    (2, 2, 40, 5000, 64, "bf16", False, 0), (1, 2, 8, 257, 128, "fp16", True, 64),
    # several query tiles of 128 rows
    (1, 2, 64, 3333, 128, "bf16", True, 0), (1, 2, 128, 1000, 64, "fp16", False, 0),
    (1, 1, 129, 4097, 128, "bf16", True, 0), (2, 1, 200, 1500, 128, "fp16", True, 3),
    (1, 2, 9, 130, 64, "bf16", False, 0), (1, 2, 100, 100, 128, "bf16", True, 1),
    # head dimension 256
    (1, 2, 1, 3000, 256, "bf16", True, 0), (1, 2, 4, 999, 256, "fp16", False, 5), (1, 1, 20, 700, 256, "bf16", True, 0),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,causal,splits", CASES)
def test_decode_matches_oracle(B, H, Nq, Nk, d, dtype, causal, splits):
    q, k, v = _inputs(B, H, Nq, Nk, d, dtype, seed=Nq * 7 + Nk)
    dev = torch.device("cuda:0")
    o, lse = fa.forward_decode(q.to(dev), k.to(dev), v.to(dev), causal=causal, num_splits=splits)
    fa.fa_device_status()
    eo, el = _check(q, k, v, o.cpu(), lse.cpu(), causal)
    assert eo <= O_TOL[dtype] and el <= LSE_TOL, (eo, el)


def test_decode_square_equals_forward():
    """With Nq = Nk the split-KV path computes what fa_forward computes."""
    q, k, v, _ = attention_inputs(1, 4, 512, 128, "bf16", seed=9, with_do=False)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    for causal in (False, True):
        o1, l1 = fa.forward(qd, kd, vd, causal=causal)
        o2, l2 = fa.forward_decode(qd, kd, vd, causal=causal, num_splits=5)
        fa.fa_device_status()
        assert float((o1.float() - o2.float()).abs().max()) <= 2 * O_TOL["bf16"]
        assert float((l1 - l2).abs().max()) <= LSE_TOL


def test_decode_full_size_sampled_heads():
    """Decode workload D1: B=4, H=32, one query, Nk=32768, d=128, bf16, causal."""
    from exact_io_aware_forward_gb300.synth import D1, decode_inputs
    q, k, v = decode_inputs(D1)
    dev = torch.device("cuda:0")
    o, lse = fa.forward_decode(q.to(dev), k.to(dev), v.to(dev), causal=True)
    fa.fa_device_status()
    eo, el = _check(q, k, v, o.cpu(), lse.cpu(), True, heads=[(0, 0), (1, 17), (3, 31)])
    assert eo <= O_TOL["bf16"] and el <= LSE_TOL, (eo, el)


@pytest.mark.parametrize("nq", [16, 64])
def test_decode_full_size_several_queries(nq):
    """The D1 shape (B=4, H=32, Nk=32768, d=128, bf16, causal) with 16 and 64
    queries per head (the tensor-core split kernel), on sampled heads."""
    import dataclasses

    from exact_io_aware_forward_gb300.synth import D1, decode_inputs
    w = dataclasses.replace(D1, Nq=nq, name=f"D1 Nq={nq}")
    q, k, v = decode_inputs(w)
    dev = torch.device("cuda:0")
    o, lse = fa.forward_decode(q.to(dev), k.to(dev), v.to(dev), causal=True)
    fa.fa_device_status()
    eo, el = _check(q, k, v, o.cpu(), lse.cpu(), True, heads=[(0, 0), (2, 9), (3, 31)])
    assert eo <= O_TOL["bf16"] and el <= LSE_TOL, (eo, el)


GQA_CASES = [  # B, Hq, Hkv, Nq, Nk, d, dtype, causal, splits
    (1, 8, 2, 1, 3000, 128, "bf16", True, 0), (2, 8, 1, 3, 1000, 64, "fp16", True, 7),
    (1, 16, 4, 16, 2000, 128, "bf16", True, 0), (1, 12, 3, 40, 700, 256, "bf16", True, 0),
    (1, 4, 2, 100, 100, 128, "fp16", False, 3), (1, 6, 6, 5, 500, 64, "bf16", True, 0),
    (2, 32, 4, 1, 4097, 256, "fp16", True, 0),
]


def _gqa_inputs(B, Hq, Hkv, Nq, Nk, d, dtype, seed):
    q, _, _, _ = attention_inputs(B, Hq, Nq, d, dtype, seed=seed, with_do=False)
    _, k, v, _ = attention_inputs(B, Hkv, Nk, d, dtype, seed=seed + 1, with_do=False)
    return q, k, v


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,dtype,causal,splits", GQA_CASES)
def test_grouped_query_decode_matches_oracle(B, Hq, Hkv, Nq, Nk, d, dtype, causal, splits):
    """Query head h against K / V head h // (Hq // Hkv): each head as its own
    rectangular problem in the oracle (tiles of 128 rows span several query
    heads on the GPU; the causal position of a row is its query index)."""
    q, k, v = _gqa_inputs(B, Hq, Hkv, Nq, Nk, d, dtype, seed=31 * Hq + Nq)
    dev = torch.device("cuda:0")
    o, lse = fa.forward_decode(q.to(dev), k.to(dev), v.to(dev), causal=causal, num_splits=splits)
    fa.fa_device_status()
    g = Hq // Hkv
    s = 1.0 / math.sqrt(d)
    qf, kf, vf = as_float64(q, k, v)
    of, lf = o.cpu().double().numpy(), lse.cpu().double().numpy()
    eo = el = 0.0
    for b in range(B):
        for h in range(Hq):
            ro, rl = A.forward_head(qf[b, h], kf[b, h // g], vf[b, h // g], s, causal)
            eo = max(eo, float(np.abs(of[b, h] - ro).max()))
            el = max(el, float(np.abs(lf[b, h] - rl).max()))
    assert eo <= O_TOL[dtype] and el <= LSE_TOL, (eo, el)


def test_grouped_query_decode_equals_repeated_heads():
    """With the same key chunks, grouped queries give bit for bit what plain
    decoding gives with every K / V head repeated for its query heads."""
    B, Hq, Hkv, Nq, Nk, d = 2, 8, 2, 7, 2500, 128
    dev = torch.device("cuda:0")
    q, k, v = (x.to(dev) for x in _gqa_inputs(B, Hq, Hkv, Nq, Nk, d, "bf16", seed=77))
    o1, l1 = fa.forward_decode(q, k, v, causal=True, num_splits=3)
    kr, vr = (x.repeat_interleave(Hq // Hkv, dim=1).contiguous() for x in (k, v))
    o2, l2 = fa.forward_decode(q, kr, vr, causal=True, num_splits=3)
    fa.fa_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)

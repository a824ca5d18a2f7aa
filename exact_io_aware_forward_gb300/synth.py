"""Seeded synthetic inputs for exact attention.

This module only draws random tensors; it holds none of the attention
arithmetic.  Both the CUDA path (tests, bench) and the float64 oracle take
their inputs from here, so the two sides always see the same values.

Two recipes:

* ``attention_inputs`` -- the workload shapes used for the GPU path:
  Q, K, V and dO i.i.d. N(0, 1) in float32, drawn in that order from
  ``torch.Generator('cpu').manual_seed(seed)``, then rounded to fp16/bf16.
  With ``k_row_scale=True`` every K row (per batch, head and position) is
  multiplied by a factor drawn from U(0.5, 3) *before* the rounding, which
  widens the range of the scores and exercises the online rescale.  The
  factor tensor is drawn after V and before dO.
* ``page_inputs`` -- the float64 workload of the tutorial page
  "FlashAttention 为什么不需要存下注意力矩阵" (jefxiong.cn), section 04:
  ``numpy.random.default_rng(seed).normal(size=(N, D))`` drawn three times
  for Q, K, V of one head.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, dtype, mask and seed."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str
    causal: bool
    seed: int
    k_row_scale: bool = False
    backward: bool = True

    @property
    def heads(self) -> int:
        return self.B * self.H

    def fwd_flops(self) -> float:
        """4*B*H*N^2*d, halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f


# The five workloads the path is specified on (shapes, dtypes, masks).
C1 = Workload("C1 fwd non-causal N=256 d=64 fp16", 1, 1, 256, 64, "fp16", False, 0, backward=False)
C2 = Workload("C2 fwd+bwd causal N=1024 d=64 fp16", 4, 16, 1024, 64, "fp16", True, 1)
C3N = Workload("C3 fwd+bwd non-causal N=4096 d=64 bf16 K-row-scaled", 2, 16, 4096, 64, "bf16", False, 2, True)
C3C = Workload("C3 fwd+bwd causal N=4096 d=64 bf16 K-row-scaled", 2, 16, 4096, 64, "bf16", True, 2, True)
C4 = Workload("C4 fwd+bwd causal N=8192 d=128 bf16", 2, 32, 8192, 128, "bf16", True, 3)
C5 = Workload("C5 fwd+bwd causal N=32768 d=128 bf16", 1, 8, 32768, 128, "bf16", True, 4)
# The long causal training shape at the widest head dimension (same B*H*d as C4).
W256 = Workload("W256 fwd+bwd causal N=8192 d=256 bf16", 2, 16, 8192, 256, "bf16", True, 9)
# d = 96 at the C4 shape.
W96 = Workload("W96 fwd+bwd causal N=8192 d=96 bf16", 2, 32, 8192, 96, "bf16", True, 10)
WORKLOADS = {"C1": C1, "C2": C2, "C3N": C3N, "C3C": C3C, "C4": C4, "C5": C5, "W256": W256, "W96": W96}


def attention_inputs(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0,
                     k_row_scale: bool = False, with_do: bool = True):
    """Return (q, k, v, do) CPU tensors of shape [B, H, N, d] in ``dtype``.

    ``do`` is None when ``with_do`` is False.  The draws are made in float32
    and rounded once to the 16-bit type (round to nearest even).
    """
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {sorted(DTYPES)}, got {dtype!r}")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if k_row_scale:
        factor = torch.rand((B, H, N, 1), generator=g, dtype=torch.float32) * 2.5 + 0.5
        k = k * factor
    do = torch.randn(shape, generator=g, dtype=torch.float32) if with_do else None
    t = DTYPES[dtype]
    return (q.to(t), k.to(t), v.to(t), None if do is None else do.to(t))


def device_inputs(B: int, H: int, N: int, d: int, dtype: str, seed: int, device, count: int = 3):
    """`count` tensors [B, H, N, d] drawn N(0,1) in float32 by a seeded
    generator on `device` and rounded once to the 16-bit type; for problems
    too large to draw on the host (the draws differ from ``attention_inputs``)."""
    g = torch.Generator(device=device).manual_seed(seed)
    return tuple(torch.randn(B, H, N, d, generator=g, device=device).to(DTYPES[dtype]) for _ in range(count))


def workload_inputs(w: Workload, with_do: bool | None = None):
    """Inputs of a named workload (see ``WORKLOADS``)."""
    if with_do is None:
        with_do = w.backward
    return attention_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, w.k_row_scale, with_do)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """Few queries (the last Nq positions) against Nk keys per head."""

    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str
    causal: bool
    seed: int

    def kv_bytes(self) -> int:
        return 2 * self.B * self.H * self.Nk * self.d * 2


# Decoding workload at the long end of the specified sequence range.
D1 = DecodeWorkload("D1 decode causal Nq=1 Nk=32768 d=128 bf16", 4, 32, 1, 32768, 128, "bf16", True, 6)


def decode_inputs(w: DecodeWorkload):
    """(q [B,H,Nq,d], k, v [B,H,Nk,d]) drawn like ``attention_inputs``."""
    q, _, _, _ = attention_inputs(w.B, w.H, w.Nq, w.d, w.dtype, seed=w.seed, with_do=False)
    _, k, v, _ = attention_inputs(w.B, w.H, w.Nk, w.d, w.dtype, seed=w.seed + 1, with_do=False)
    return q, k, v


@dataclasses.dataclass(frozen=True)
class BlockSparseWorkload:
    """Attention restricted to the kept 128 x 128 blocks of a block mask."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str
    causal: bool
    density: float  # probability that an off-diagonal block is kept
    per_head: bool  # one mask per (b, h) head, else one mask for all heads
    seed: int

    @property
    def tiles(self) -> int:
        return (self.N + 127) // 128


def block_mask(w: BlockSparseWorkload) -> np.ndarray:
    """Boolean mask [1 or B*H, T, T], T = ceil(N/128): each block kept with
    probability ``density``, the diagonal block always kept, drawn from
    ``numpy.random.default_rng(seed)``."""
    T = w.tiles
    rng = np.random.default_rng(w.seed)
    bm = rng.random((w.B * w.H if w.per_head else 1, T, T)) < w.density
    bm[:, np.arange(T), np.arange(T)] = True
    return bm


# Block-sparse workload: the shape of the long causal training problem with a
# random half of the off-diagonal blocks kept, one mask shared by all heads.
S1 = BlockSparseWorkload("S1 block-sparse density 0.5 N=8192 d=128 bf16", 2, 32, 8192, 128, "bf16", False, 0.5,
                         False, 7)


def blocksparse_inputs(w: BlockSparseWorkload):
    """(q, k, v, dO [B,H,N,d], mask [1 or B*H, T, T] bool)."""
    q, k, v, do = attention_inputs(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed)
    return q, k, v, do, block_mask(w)


@dataclasses.dataclass(frozen=True)
class VarlenWorkload:
    """A packed batch of sequences of different lengths (query = key lengths)."""

    name: str
    H: int
    d: int
    dtype: str
    causal: bool
    lengths: tuple
    seed: int

    @property
    def B(self) -> int:
        return len(self.lengths)


def _lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    return tuple(int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, size=n))


# Variable-length workload: 16 causal sequences of 256 .. 8192 tokens (uniform), the
# head shape of the long training problem.
V1 = VarlenWorkload("V1 varlen 16 seqs of 256-8192 tokens H=32 d=128 bf16 causal", 32, 128, "bf16", True,
                    _lengths(16, 256, 8192, 8), 8)


def varlen_workload_inputs(w: VarlenWorkload):
    return varlen_inputs(w.lengths, w.lengths, w.H, w.d, w.dtype, w.seed)


def varlen_inputs(lengths_q, lengths_k, H: int, d: int, dtype: str, seed: int, with_do: bool = True):
    """Packed token-major q, dO [sum(lengths_q), H, d], k, v [sum(lengths_k), H, d]
    (16-bit, N(0,1) before rounding, drawn in that order from one generator)
    and the int32 offsets cu_q, cu_k (B + 1 entries each)."""
    g = torch.Generator().manual_seed(seed)
    dt = DTYPES[dtype]
    Tq, Tk = int(sum(lengths_q)), int(sum(lengths_k))
    q = torch.randn(Tq, H, d, generator=g).to(dt)
    k = torch.randn(Tk, H, d, generator=g).to(dt)
    v = torch.randn(Tk, H, d, generator=g).to(dt)
    do = torch.randn(Tq, H, d, generator=g).to(dt) if with_do else None
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lengths_q)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lengths_k)]), dtype=torch.int32)
    return q, k, v, do, cu_q, cu_k


def page_inputs(N: int, D: int, seed: int):
    """float64 Q, K, V of one head, drawn like the tutorial page's demos."""
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(N, D))
    k = rng.normal(size=(N, D))
    v = rng.normal(size=(N, D))
    return q, k, v


def as_float64(*tensors):
    """Exact upcast of 16-bit tensors to float64 numpy arrays (None passes)."""
    return tuple(None if t is None else t.to(torch.float64).numpy() for t in tensors)

"""Python binding of the C ABI in ``include/fa_gb300.h``.

Argument marshalling only: the functions named like the C entry points take
torch CUDA tensors, check dtype/shape/contiguity, and pass raw device
pointers plus the current CUDA stream to the library.  Every step of the
computation runs in the library's kernels.  ``forward`` and ``backward`` are
conveniences that also allocate the outputs (and the backward workspace)
with torch.
"""
from __future__ import annotations

import ctypes
import math

import torch

from ._lib import lib, status_string

FA_FP16, FA_BF16 = 0, 1
_DTYPE_CODE = {torch.float16: FA_FP16, torch.bfloat16: FA_BF16}


class FAError(RuntimeError):
    """A non-zero fa_status returned by the library."""

    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code}: {status_string(code)}")
        self.code = code


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise FAError(fn, code)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes_stream(stream)


def ctypes_stream(stream) -> int:
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _bhnd(name, t, like=None, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [B, H, N, d]")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if like is not None and tuple(t.shape) != tuple(like):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(like)}")
    return t.data_ptr()


def _shape(q):
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    if q.dtype not in _DTYPE_CODE:
        raise TypeError("q must be float16 or bfloat16")
    return tuple(q.shape)


def _scale(scale, d):
    return float(1.0 / math.sqrt(d) if scale is None else scale)


# ---------------------------------------------------------------- C entry points
def fa_forward(q, k, v, o, lse, causal=False, scale=None, stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt),
            _bhnd("o", o, q.shape, dt), _bhnd("lse", lse, (B, H, N), torch.float32)]
    _check("fa_forward", lib().fa_forward(*args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)),
                                          _scale(scale, d), _stream(stream)))


def _block_mask(block_mask, B, H, N):
    T = (N + 127) // 128
    if not isinstance(block_mask, torch.Tensor) or not block_mask.is_cuda or block_mask.dtype != torch.uint8:
        raise TypeError("block_mask must be a CUDA uint8 tensor")
    if not block_mask.is_contiguous() or block_mask.dim() != 3 or tuple(block_mask.shape[1:]) != (T, T) \
            or block_mask.shape[0] not in (1, B * H):
        raise ValueError(f"block_mask must be contiguous [1 or B*H, {T}, {T}]")
    return block_mask.data_ptr(), int(block_mask.shape[0])


def fa_forward_blocksparse(q, k, v, o, lse, block_mask, causal=False, scale=None, stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    mptr, mheads = _block_mask(block_mask, B, H, N)
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt),
            _bhnd("o", o, q.shape, dt), _bhnd("lse", lse, (B, H, N), torch.float32)]
    _check("fa_forward_blocksparse", lib().fa_forward_blocksparse(*args, mptr, mheads, B, H, N, d, _DTYPE_CODE[dt],
                                                                  int(bool(causal)), _scale(scale, d),
                                                                  _stream(stream)))


def fa_backward_blocksparse(q, k, v, o, do, lse, dq, dk, dv, block_mask, workspace, causal=False, scale=None,
                            stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    mptr, mheads = _block_mask(block_mask, B, H, N)
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("o", o, q.shape, dt),
            _bhnd("do", do, q.shape, dt), _bhnd("lse", lse, (B, H, N), torch.float32),
            _bhnd("dq", dq, q.shape, dt), _bhnd("dk", dk, q.shape, dt), _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_blocksparse", lib().fa_backward_blocksparse(
        *args, mptr, mheads, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), workspace.data_ptr(),
        workspace.numel(), _stream(stream)))


def _seed_offset(seed, offset):
    seed, offset = int(seed), int(offset)
    if not (0 <= seed < 2**64 and 0 <= offset < 2**32):
        raise ValueError("seed must fit 64 bits and offset 32 bits (unsigned)")
    return seed, offset


def fa_forward_dropout(q, k, v, o, lse, p_drop, seed, offset, causal=False, scale=None, stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    seed, offset = _seed_offset(seed, offset)
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt),
            _bhnd("o", o, q.shape, dt), _bhnd("lse", lse, (B, H, N), torch.float32)]
    _check("fa_forward_dropout", lib().fa_forward_dropout(*args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)),
                                                          _scale(scale, d), float(p_drop), seed, offset,
                                                          _stream(stream)))


def fa_backward_dropout(q, k, v, o, do, lse, dq, dk, dv, workspace, p_drop, seed, offset, causal=False, scale=None,
                        stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    seed, offset = _seed_offset(seed, offset)
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("o", o, q.shape, dt),
            _bhnd("do", do, q.shape, dt), _bhnd("lse", lse, (B, H, N), torch.float32),
            _bhnd("dq", dq, q.shape, dt), _bhnd("dk", dk, q.shape, dt), _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_dropout", lib().fa_backward_dropout(
        *args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), float(p_drop), seed, offset,
        workspace.data_ptr(), workspace.numel(), _stream(stream)))


def fa_backward_dkdv_dropout(q, k, v, do, lse, delta, dq_accum, dk, dv, p_drop, seed, offset, causal=False,
                             scale=None, stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    seed, offset = _seed_offset(seed, offset)
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dq_accum", dq_accum, q.shape, torch.float32), _bhnd("dk", dk, q.shape, dt),
            _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_dkdv_dropout", lib().fa_backward_dkdv_dropout(
        *args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), float(p_drop), seed, offset,
        _stream(stream)))


def fa_backward_dk_dv_dropout(q, k, v, do, lse, delta, dk, dv, p_drop, seed, offset, causal=False, scale=None,
                              stream=None) -> None:
    """Split backward with dropout: dK and dV."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    seed, offset = _seed_offset(seed, offset)
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dk", dk, q.shape, dt), _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_dk_dv_dropout", lib().fa_backward_dk_dv_dropout(
        *args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), float(p_drop), seed, offset,
        _stream(stream)))


def fa_backward_dq_dropout(q, k, v, do, lse, delta, dq, p_drop, seed, offset, causal=False, scale=None,
                           stream=None) -> None:
    """Split backward with dropout: dQ."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    seed, offset = _seed_offset(seed, offset)
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dq", dq, q.shape, dt)]
    _check("fa_backward_dq_dropout", lib().fa_backward_dq_dropout(
        *args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), float(p_drop), seed, offset,
        _stream(stream)))


def fa_dropout_keep_mask(keep, p_drop, seed, offset, stream=None) -> None:
    """Write the keep mask ([BH, Nq, Nk] uint8 CUDA tensor, 1 = kept) the dropout entry points use."""
    if not isinstance(keep, torch.Tensor) or not keep.is_cuda or keep.dtype != torch.uint8 \
            or not keep.is_contiguous() or keep.dim() != 3:
        raise TypeError("keep must be a contiguous CUDA uint8 tensor [BH, Nq, Nk]")
    seed, offset = _seed_offset(seed, offset)
    BH, Nq, Nk = keep.shape
    _check("fa_dropout_keep_mask", lib().fa_dropout_keep_mask(keep.data_ptr(), BH, Nq, Nk, float(p_drop), seed,
                                                              offset, _stream(stream)))


# ---------------------------------------------------------------- packed variable-length batches
def _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k):
    if q.dim() != 3 or k.dim() != 3 or q.shape[1:] != k.shape[1:]:
        raise ValueError("q must be [total_q, H, d] and k, v [total_k, H, d]")
    if q.dtype not in _DTYPE_CODE:
        raise TypeError("q must be float16 or bfloat16")
    for name, cu in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if not isinstance(cu, torch.Tensor) or not cu.is_cuda or cu.dtype != torch.int32 or not cu.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA int32 tensor")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 offsets")
    B = cu_seqlens_q.numel() - 1
    Tq, H, d = q.shape
    return B, H, d, Tq, k.shape[0]


def fa_forward_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False,
                      scale=None, dropout_p=0.0, seed=0, offset=0, stream=None) -> None:
    B, H, d, Tq, Tk = _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k)
    dt = q.dtype
    seed, offset = _seed_offset(seed, offset)
    args = [_bhnd("q", q), _bhnd("k", k, k.shape, dt), _bhnd("v", v, k.shape, dt), _bhnd("o", o, q.shape, dt),
            _bhnd("lse", lse, (Tq, H), torch.float32), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr()]
    _check("fa_forward_varlen", lib().fa_forward_varlen(
        *args, B, H, int(max_seqlen_q), int(max_seqlen_k), Tq, Tk, d, _DTYPE_CODE[dt], int(bool(causal)),
        _scale(scale, d), float(dropout_p), seed, offset, _stream(stream)))


def fa_backward_varlen_workspace_size(total_q, H, d) -> int:
    return int(lib().fa_backward_varlen_workspace_size(int(total_q), int(H), int(d)))


def fa_backward_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                       workspace, causal=False, scale=None, dropout_p=0.0, seed=0, offset=0, stream=None) -> None:
    B, H, d, Tq, Tk = _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k)
    dt = q.dtype
    seed, offset = _seed_offset(seed, offset)
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    args = [_bhnd("q", q), _bhnd("k", k, k.shape, dt), _bhnd("v", v, k.shape, dt), _bhnd("o", o, q.shape, dt),
            _bhnd("do", do, q.shape, dt), _bhnd("lse", lse, (Tq, H), torch.float32), _bhnd("dq", dq, q.shape, dt),
            _bhnd("dk", dk, k.shape, dt), _bhnd("dv", dv, k.shape, dt), cu_seqlens_q.data_ptr(),
            cu_seqlens_k.data_ptr()]
    _check("fa_backward_varlen", lib().fa_backward_varlen(
        *args, B, H, int(max_seqlen_q), int(max_seqlen_k), Tq, Tk, d, _DTYPE_CODE[dt], int(bool(causal)),
        _scale(scale, d), float(dropout_p), seed, offset, workspace.data_ptr(), workspace.numel(), _stream(stream)))


def fa_backward_dkdv_varlen(q, k, v, do, lse, delta, dq_accum, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                            max_seqlen_k, causal=False, scale=None, dropout_p=0.0, seed=0, offset=0,
                            stream=None) -> None:
    B, H, d, Tq, Tk = _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k)
    dt = q.dtype
    seed, offset = _seed_offset(seed, offset)
    args = [_bhnd("q", q), _bhnd("k", k, k.shape, dt), _bhnd("v", v, k.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (Tq, H), torch.float32), _bhnd("delta", delta, (Tq, H), torch.float32),
            _bhnd("dq_accum", dq_accum, q.shape, torch.float32), _bhnd("dk", dk, k.shape, dt),
            _bhnd("dv", dv, k.shape, dt), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr()]
    _check("fa_backward_dkdv_varlen", lib().fa_backward_dkdv_varlen(
        *args, B, H, int(max_seqlen_q), int(max_seqlen_k), Tq, Tk, d, _DTYPE_CODE[dt], int(bool(causal)),
        _scale(scale, d), float(dropout_p), seed, offset, _stream(stream)))


def fa_backward_dk_dv_varlen(q, k, v, do, lse, delta, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                             max_seqlen_k, causal=False, scale=None, stream=None) -> None:
    """Split backward of a packed batch: dK and dV (no dQ work)."""
    B, H, d, Tq, Tk = _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k)
    dt = q.dtype
    args = [_bhnd("q", q), _bhnd("k", k, k.shape, dt), _bhnd("v", v, k.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (Tq, H), torch.float32), _bhnd("delta", delta, (Tq, H), torch.float32),
            _bhnd("dk", dk, k.shape, dt), _bhnd("dv", dv, k.shape, dt), cu_seqlens_q.data_ptr(),
            cu_seqlens_k.data_ptr()]
    _check("fa_backward_dk_dv_varlen", lib().fa_backward_dk_dv_varlen(
        *args, B, H, int(max_seqlen_q), int(max_seqlen_k), Tq, Tk, d, _DTYPE_CODE[dt], int(bool(causal)),
        _scale(scale, d), _stream(stream)))


def fa_backward_dq_varlen(q, k, v, do, lse, delta, dq, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                          causal=False, scale=None, stream=None) -> None:
    """Split backward of a packed batch: dQ by its own kernel."""
    B, H, d, Tq, Tk = _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k)
    dt = q.dtype
    args = [_bhnd("q", q), _bhnd("k", k, k.shape, dt), _bhnd("v", v, k.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (Tq, H), torch.float32), _bhnd("delta", delta, (Tq, H), torch.float32),
            _bhnd("dq", dq, q.shape, dt), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr()]
    _check("fa_backward_dq_varlen", lib().fa_backward_dq_varlen(
        *args, B, H, int(max_seqlen_q), int(max_seqlen_k), Tq, Tk, d, _DTYPE_CODE[dt], int(bool(causal)),
        _scale(scale, d), _stream(stream)))


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False, scale=None,
                   dropout_p=0.0, seed=0, offset=0, stream=None):
    """Return (O [total_q, H, d], LSE [total_q, H]) for packed sequences."""
    o = torch.empty_like(q)
    lse = torch.empty((q.shape[0], q.shape[1]), device=q.device, dtype=torch.float32)
    fa_forward_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, scale,
                      dropout_p, seed, offset, stream)
    return o, lse


def backward_varlen(q, k, v, o, lse, do, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=False,
                    scale=None, dropout_p=0.0, seed=0, offset=0, stream=None, workspace=None):
    """Return (dQ, dK, dV) for packed sequences (same arguments as the forward)."""
    if workspace is None:
        n = fa_backward_varlen_workspace_size(q.shape[0], q.shape[1], q.shape[2])
        workspace = torch.empty(max(n, 1), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_backward_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                       workspace, causal, scale, dropout_p, seed, offset, stream)
    return dq, dk, dv


def fa_backward_workspace_size(B, H, N, d) -> int:
    return int(lib().fa_backward_workspace_size(B, H, N, d))


def fa_backward(q, k, v, o, do, lse, dq, dk, dv, workspace, causal=False, scale=None, stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("o", o, q.shape, dt),
            _bhnd("do", do, q.shape, dt), _bhnd("lse", lse, (B, H, N), torch.float32),
            _bhnd("dq", dq, q.shape, dt), _bhnd("dk", dk, q.shape, dt), _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward", lib().fa_backward(*args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)),
                                            _scale(scale, d), workspace.data_ptr(), workspace.numel(),
                                            _stream(stream)))


def fa_backward_noalloc(q, k, v, o, do, lse, dq, dk, dv, causal=False, scale=None, stream=None) -> None:
    """fa_backward without a workspace: the library's fixed device scratch
    (32 MiB per GPU) holds D and the dQ accumulator.  For callers that cannot
    allocate device memory.  Calls that overlap on the GPU share that scratch
    and must be serialised; the first call on a device must precede any
    stream capture."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("o", o, q.shape, dt),
            _bhnd("do", do, q.shape, dt), _bhnd("lse", lse, (B, H, N), torch.float32),
            _bhnd("dq", dq, q.shape, dt), _bhnd("dk", dk, q.shape, dt), _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_noalloc", lib().fa_backward_noalloc(*args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)),
                                                            _scale(scale, d), _stream(stream)))


def fa_backward_preprocess(o, do, delta, dq_accum, stream=None) -> None:
    """D = rowsum(dO * O) into ``delta``; ``dq_accum`` zeroed, or None (D only)."""
    B, H, N, d = _shape(o)
    dt = o.dtype
    args = [_bhnd("o", o), _bhnd("do", do, o.shape, dt), _bhnd("delta", delta, (B, H, N), torch.float32),
            None if dq_accum is None else _bhnd("dq_accum", dq_accum, o.shape, torch.float32)]
    _check("fa_backward_preprocess",
           lib().fa_backward_preprocess(*args, B, H, N, d, _DTYPE_CODE[dt], _stream(stream)))


def fa_backward_dkdv(q, k, v, do, lse, delta, dq_accum, dk, dv, causal=False, scale=None, stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dq_accum", dq_accum, q.shape, torch.float32), _bhnd("dk", dk, q.shape, dt),
            _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_dkdv", lib().fa_backward_dkdv(*args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)),
                                                      _scale(scale, d), _stream(stream)))


def fa_backward_dkdv_blocksparse(q, k, v, do, lse, delta, dq_accum, dk, dv, block_mask, causal=False, scale=None,
                                 stream=None) -> None:
    B, H, N, d = _shape(q)
    dt = q.dtype
    mptr, mheads = _block_mask(block_mask, B, H, N)
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dq_accum", dq_accum, q.shape, torch.float32), _bhnd("dk", dk, q.shape, dt),
            _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_dkdv_blocksparse", lib().fa_backward_dkdv_blocksparse(
        *args, mptr, mheads, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), _stream(stream)))


def fa_backward_dk_dv(q, k, v, do, lse, delta, dk, dv, causal=False, scale=None, stream=None) -> None:
    """Split backward: dK and dV (no dQ work)."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dk", dk, q.shape, dt), _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_dk_dv", lib().fa_backward_dk_dv(*args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)),
                                                        _scale(scale, d), _stream(stream)))


def fa_backward_dq(q, k, v, do, lse, delta, dq, causal=False, scale=None, stream=None) -> None:
    """Split backward: dQ by its own kernel (recomputes P and dP)."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dq", dq, q.shape, dt)]
    _check("fa_backward_dq", lib().fa_backward_dq(*args, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)),
                                                  _scale(scale, d), _stream(stream)))


def fa_backward_dk_dv_blocksparse(q, k, v, do, lse, delta, dk, dv, block_mask, causal=False, scale=None,
                                  stream=None) -> None:
    """Split backward restricted to the kept blocks: dK and dV."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    mptr, mheads = _block_mask(block_mask, B, H, N)
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dk", dk, q.shape, dt), _bhnd("dv", dv, q.shape, dt)]
    _check("fa_backward_dk_dv_blocksparse", lib().fa_backward_dk_dv_blocksparse(
        *args, mptr, mheads, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), _stream(stream)))


def fa_backward_dq_blocksparse(q, k, v, do, lse, delta, dq, block_mask, causal=False, scale=None,
                               stream=None) -> None:
    """Split backward restricted to the kept blocks: dQ."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    mptr, mheads = _block_mask(block_mask, B, H, N)
    args = [_bhnd("q", q), _bhnd("k", k, q.shape, dt), _bhnd("v", v, q.shape, dt), _bhnd("do", do, q.shape, dt),
            _bhnd("lse", lse, (B, H, N), torch.float32), _bhnd("delta", delta, (B, H, N), torch.float32),
            _bhnd("dq", dq, q.shape, dt)]
    _check("fa_backward_dq_blocksparse", lib().fa_backward_dq_blocksparse(
        *args, mptr, mheads, B, H, N, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), _stream(stream)))


def fa_backward_dq_convert(dq_accum, dq, scale=None, stream=None) -> None:
    B, H, N, d = _shape(dq)
    args = [_bhnd("dq_accum", dq_accum, dq.shape, torch.float32), _bhnd("dq", dq)]
    _check("fa_backward_dq_convert", lib().fa_backward_dq_convert(*args, B, H, N, d, _DTYPE_CODE[dq.dtype],
                                                                  _scale(scale, d), _stream(stream)))


def fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits=0) -> int:
    return int(lib().fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits))


def fa_forward_decode(q, k, v, o, lse, workspace, causal=False, scale=None, num_splits=0, stream=None) -> None:
    """Split-KV forward: q, o [B,H,Nq,d]; k, v [B,H,Nk,d]; lse [B,H,Nq]."""
    B, H, Nq, d = _shape(q)
    dt = q.dtype
    if k.dim() != 4 or k.shape[:2] != q.shape[:2] or k.shape[3] != d:
        raise ValueError("k must be [B, H, Nk, d] with q's B, H, d")
    Nk = k.shape[2]
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    args = [_bhnd("q", q), _bhnd("k", k, None, dt), _bhnd("v", v, k.shape, dt), _bhnd("o", o, q.shape, dt),
            _bhnd("lse", lse, (B, H, Nq), torch.float32)]
    _check("fa_forward_decode", lib().fa_forward_decode(*args, B, H, Nq, Nk, d, _DTYPE_CODE[dt], int(bool(causal)),
                                                        _scale(scale, d), int(num_splits), workspace.data_ptr(),
                                                        workspace.numel(), _stream(stream)))


def fa_decode_gqa_workspace_size(B, Hq, Hkv, Nq, Nk, d, num_splits=0) -> int:
    return int(lib().fa_decode_gqa_workspace_size(B, Hq, Hkv, Nq, Nk, d, num_splits))


def fa_forward_decode_gqa(q, k, v, o, lse, workspace, causal=False, scale=None, num_splits=0, stream=None) -> None:
    """Split-KV forward with grouped queries: q, o [B,Hq,Nq,d]; k, v [B,Hkv,Nk,d]
    (Hq a multiple of Hkv; query head h reads K / V head h // (Hq // Hkv)); lse [B,Hq,Nq]."""
    B, Hq, Nq, d = _shape(q)
    dt = q.dtype
    if k.dim() != 4 or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k must be [B, Hkv, Nk, d] with q's B and d")
    Hkv, Nk = k.shape[1], k.shape[2]
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA uint8 tensor")
    args = [_bhnd("q", q), _bhnd("k", k, None, dt), _bhnd("v", v, k.shape, dt), _bhnd("o", o, q.shape, dt),
            _bhnd("lse", lse, (B, Hq, Nq), torch.float32)]
    _check("fa_forward_decode_gqa", lib().fa_forward_decode_gqa(
        *args, B, Hq, Hkv, Nq, Nk, d, _DTYPE_CODE[dt], int(bool(causal)), _scale(scale, d), int(num_splits),
        workspace.data_ptr(), workspace.numel(), _stream(stream)))


def fa_selftest_wait_timeout(stream=None) -> None:
    """Enqueue the failure-detection self-test (a bounded wait that never
    completes; ~2 s); the next fa_device_status() raises FA_ERR_TIMEOUT."""
    _check("fa_selftest_wait_timeout", lib().fa_selftest_wait_timeout(_stream(stream)))


def fa_device_status(stream=None) -> None:
    """Synchronise ``stream``; raise FAError if a kernel latched a timeout."""
    _check("fa_device_status", lib().fa_device_status(_stream(stream)))


def fa_score_blocks(reset=False, stream=None):
    """Synchronise ``stream``; return (forward, backward) counts of the 64 x 64
    score blocks the kernels computed since the last reset (and reset them
    if ``reset``)."""
    f, b = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check("fa_score_blocks", lib().fa_score_blocks(_stream(stream), ctypes.byref(f), ctypes.byref(b), int(bool(reset))))
    return f.value, b.value


# ---------------------------------------------------------------- conveniences
def forward(q, k, v, causal=False, scale=None, stream=None, block_mask=None, dropout_p=0.0, seed=0, offset=0):
    """Return (O, LSE) for [B, H, N, d] q, k, v (block-sparse if block_mask is
    given; with dropout on P if dropout_p > 0, keep mask drawn from seed and offset)."""
    B, H, N, d = _shape(q)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    if dropout_p and block_mask is not None:
        raise ValueError("dropout is supported for dense attention only")
    if dropout_p:
        fa_forward_dropout(q, k, v, o, lse, dropout_p, seed, offset, causal, scale, stream)
    elif block_mask is None:
        fa_forward(q, k, v, o, lse, causal, scale, stream)
    else:
        fa_forward_blocksparse(q, k, v, o, lse, block_mask, causal, scale, stream)
    return o, lse


def forward_decode(q, k, v, causal=False, scale=None, num_splits=0, stream=None, workspace=None):
    """Return (O, LSE) for few queries q [B,Hq,Nq,d] against k, v [B,Hkv,Nk,d]
    (Hkv = Hq, or grouped queries: Hq a multiple of Hkv)."""
    B, H, Nq, d = _shape(q)
    grouped = k.dim() == 4 and k.shape[1] != H
    if workspace is None:
        n = (fa_decode_gqa_workspace_size(B, H, k.shape[1], Nq, k.shape[2], d, num_splits) if grouped
             else fa_decode_workspace_size(B, H, Nq, k.shape[2], d, num_splits))
        workspace = torch.empty(max(n, 1), device=q.device, dtype=torch.uint8)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    if grouped:
        fa_forward_decode_gqa(q, k, v, o, lse, workspace, causal, scale, num_splits, stream)
    else:
        fa_forward_decode(q, k, v, o, lse, workspace, causal, scale, num_splits, stream)
    return o, lse


def backward(q, k, v, o, lse, do, causal=False, scale=None, stream=None, workspace=None, block_mask=None,
             dropout_p=0.0, seed=0, offset=0):
    """Return (dQ, dK, dV) (block-sparse if block_mask is given; with the
    forward's dropout if dropout_p > 0 -- pass the same seed and offset)."""
    B, H, N, d = _shape(q)
    if workspace is None:
        workspace = torch.empty(fa_backward_workspace_size(B, H, N, d), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if dropout_p and block_mask is not None:
        raise ValueError("dropout is supported for dense attention only")
    if dropout_p:
        fa_backward_dropout(q, k, v, o, do, lse, dq, dk, dv, workspace, dropout_p, seed, offset, causal, scale, stream)
    elif block_mask is None:
        fa_backward(q, k, v, o, do, lse, dq, dk, dv, workspace, causal, scale, stream)
    else:
        fa_backward_blocksparse(q, k, v, o, do, lse, dq, dk, dv, block_mask, workspace, causal, scale, stream)
    return dq, dk, dv

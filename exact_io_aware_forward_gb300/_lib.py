"""ctypes loader for ``libfa_gb300.so`` -- argument types only, no logic.

The names and signatures mirror ``include/fa_gb300.h`` one to one.
Loading fails loudly (RuntimeError) when the library has not been built;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa_gb300.so")

# Every symbol include/fa_gb300.h declares: name -> (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t
_U64 = ctypes.c_uint64
_U32 = ctypes.c_uint32
SIGNATURES = {
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_forward_blocksparse": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_backward_workspace_size": (_S, [_I, _I, _I, _I]),
    "fa_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _S, _P]),
    "fa_backward_blocksparse": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _S,
                                     _P]),
    "fa_backward_preprocess": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "fa_backward_dkdv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_backward_dkdv_blocksparse": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                          _P]),
    "fa_backward_dq_convert": (_I, [_P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "fa_backward_dk_dv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_backward_dq": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_backward_dk_dv_blocksparse": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                           _P]),
    "fa_backward_dq_blocksparse": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_backward_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_decode_workspace_size": (_S, [_I, _I, _I, _I, _I, _I]),
    "fa_forward_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "fa_decode_gqa_workspace_size": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_forward_decode_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "fa_forward_dropout": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _U64, _U32, _P]),
    "fa_backward_dropout": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _U64, _U32, _P,
                                 _S, _P]),
    "fa_backward_dkdv_dropout": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _U64, _U32,
                                      _P]),
    "fa_backward_dk_dv_dropout": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _U64, _U32,
                                       _P]),
    "fa_backward_dq_dropout": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _U64, _U32, _P]),
    "fa_dropout_keep_mask": (_I, [_P, _I, _I, _I, _F, _U64, _U32, _P]),
    "fa_forward_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _U64, _U32,
                               _P]),
    "fa_backward_varlen_workspace_size": (_S, [_I, _I, _I]),
    "fa_backward_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                                _F, _U64, _U32, _P, _S, _P]),
    "fa_backward_dkdv_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                     _I, _F, _F, _U64, _U32, _P]),
    "fa_backward_dk_dv_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                      _F, _P]),
    "fa_backward_dq_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_selftest_wait_timeout": (_I, [_P]),
    "fa_device_status": (_I, [_P]),
    "fa_score_blocks": (_I, [_P, ctypes.POINTER(_U64), ctypes.POINTER(_U64), _I]),
}

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -m exact_io_aware_forward_gb300.build` (needs nvcc)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def status_string(code: int) -> str:
    return lib().fa_status_string(int(code)).decode()

"""The C-ABI library builds, loads and exports every symbol the header
declares; argument validation rejects bad calls before any CUDA work.
No kernel is launched here (no GPU needed)."""
import os
import re

import pytest

from exact_io_aware_forward_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_gb300.h")


def _declared():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    from exact_io_aware_forward_gb300 import _lib
    return _lib.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("fa_forward", "fa_backward", "fa_backward_workspace_size", "fa_status_string",
                 "fa_device_status"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from exact_io_aware_forward_gb300 import _lib
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    from exact_io_aware_forward_gb300._lib import status_string
    assert status_string(0) == "FA_OK"
    for code in range(1, 6):
        assert status_string(code).startswith("FA_ERR_")
    assert status_string(99) == "unknown fa_status"


def test_workspace_size_is_linear_in_n(lib):
    ws = lib.fa_backward_workspace_size
    assert ws(1, 1, 0, 64) == 0 and ws(1, 1, 16, 80) == 0 and ws(1, 1, 16, 96) == 16 * (4 + 4 * 96) + 192
    a, b = ws(2, 32, 8192, 128), ws(2, 32, 16384, 128)
    assert a == 2 * 32 * 8192 * (4 + 4 * 128)
    assert b == 2 * a


@pytest.mark.parametrize("case", ["null", "bad_d", "bad_dtype", "bad_scale", "misaligned", "bad_n"])
def test_forward_rejects_bad_arguments(lib, case):
    ptr = 1 << 20  # aligned, never dereferenced: validation fails before any launch
    args = dict(q=ptr, k=ptr, v=ptr, o=ptr, lse=ptr, B=1, H=1, N=16, d=64, dt=1, causal=0, scale=0.125)
    want = 1
    if case == "null":
        args["q"] = None
    elif case == "bad_d":
        args["d"], want = 80, 2
    elif case == "bad_dtype":
        args["dt"], want = 7, 2
    elif case == "bad_scale":
        args["scale"] = float("nan")
    elif case == "misaligned":
        args["o"] = ptr + 2
    elif case == "bad_n":
        args["N"] = 0
    rc = lib.fa_forward(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["H"],
                        args["N"], args["d"], args["dt"], args["causal"], args["scale"], None)
    assert rc == want


def test_backward_rejects_small_workspace(lib):
    ptr = 1 << 20
    rc = lib.fa_backward(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 64, 1, 0, 0.125,
                         ptr, 16, None)
    assert rc == 5


def test_decode_workspace_and_validation(lib):
    ws = lib.fa_decode_workspace_size
    assert ws(1, 1, 1, 0, 128, 0) == 0 and ws(1, 1, 1, 100, 96, 0) == 0 and ws(1, 1, 1, 100, 128, 2000) == 0
    n = ws(1, 2, 3, 1000, 64, 4)  # 4 chunks of 256 keys, 6 rows each
    assert n == ((4 * 6 * 64 * 4 + 255) // 256) * 256 + ((4 * 6 * 4 + 255) // 256) * 256
    ptr = 1 << 20
    # causal with more queries than keys has no reading: rejected before any launch
    rc = lib.fa_forward_decode(ptr, ptr, ptr, ptr, ptr, 1, 1, 8, 4, 64, 1, 1, 0.125, 0, ptr, 1 << 20, None)
    assert rc == 1
    rc = lib.fa_forward_decode(ptr, ptr, ptr, ptr, ptr, 1, 1, 2, 4, 64, 1, 0, 0.125, 0, ptr, 16, None)
    assert rc == 5


def test_blocksparse_mask_validation(lib):
    """A null mask or a mask count that is neither 1 nor B*H is rejected
    before any launch, in all three block-sparse entry points."""
    ptr = 1 << 20
    for mask, heads in ((None, 1), (ptr, 0), (ptr, 5)):
        rc = lib.fa_forward_blocksparse(ptr, ptr, ptr, ptr, ptr, mask, heads, 2, 3, 300, 64, 1, 0, 0.125, None)
        assert rc == 1
        rc = lib.fa_backward_blocksparse(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, mask, heads, 2, 3, 300, 64, 1,
                                         0, 0.125, ptr, 1 << 30, None)
        assert rc == 1
        rc = lib.fa_backward_dkdv_blocksparse(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, mask, heads, 2, 3, 300, 64,
                                              1, 0, 0.125, None)
        assert rc == 1
    # shape errors still come first with a valid mask count
    rc = lib.fa_forward_blocksparse(ptr, ptr, ptr, ptr, ptr, ptr, 6, 2, 3, 300, 80, 1, 0, 0.125, None)
    assert rc == 2


def test_dropout_validation(lib):
    """p outside [0, 1), NaN, or rounding to 1 is rejected before any launch."""
    ptr = 1 << 20
    for p in (-0.1, 1.0, float("nan"), 1.0 - 2 ** -18):
        rc = lib.fa_forward_dropout(ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 64, 1, 0, 0.125, p, 1, 0, None)
        assert rc == 1, p
        rc = lib.fa_backward_dropout(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 64, 1, 0, 0.125, p, 1, 0,
                                     ptr, 1 << 30, None)
        assert rc == 1, p
        rc = lib.fa_backward_dkdv_dropout(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 64, 1, 0, 0.125, p,
                                          1, 0, None)
        assert rc == 1, p
        rc = lib.fa_backward_dk_dv_dropout(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 64, 1, 0, 0.125, p, 1, 0,
                                           None)
        assert rc == 1, p
        rc = lib.fa_backward_dq_dropout(ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 64, 1, 0, 0.125, p, 1, 0, None)
        assert rc == 1, p
        assert lib.fa_dropout_keep_mask(ptr, 1, 4, 4, p, 1, 0, None) == 1
    # the split dropout stages: d = 256 is unsupported, a misaligned tensor is
    # an invalid argument, both before any launch
    assert lib.fa_backward_dq_dropout(ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 256, 1, 0, 0.0625, 0.1, 1, 0,
                                      None) == 2
    assert lib.fa_backward_dk_dv_dropout(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 256, 1, 0, 0.0625, 0.1, 1,
                                         0, None) == 2
    assert lib.fa_backward_dq_dropout(ptr + 2, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 16, 64, 1, 0, 0.125, 0.1, 1, 0,
                                      None) == 1
    assert lib.fa_dropout_keep_mask(None, 1, 4, 4, 0.5, 1, 0, None) == 1
    assert lib.fa_dropout_keep_mask(ptr, 0, 4, 4, 0.5, 1, 0, None) == 1


def test_varlen_validation(lib):
    """Host-side checks of the packed variable-length entry points (the
    offsets themselves are only read on the device)."""
    ptr = 1 << 20
    good = dict(B=2, H=3, mq=100, mk=120, tq=150, tk=200, d=64)

    def fwd(cu_q=ptr, cu_k=ptr, **kw):
        a = dict(good, **kw)
        return lib.fa_forward_varlen(ptr, ptr, ptr, ptr, ptr, cu_q, cu_k, a["B"], a["H"], a["mq"], a["mk"], a["tq"],
                                     a["tk"], a["d"], 1, 1, 0.125, 0.0, 0, 0, None)

    assert fwd(cu_q=None) == 1 and fwd(cu_k=ptr + 2) == 1
    assert fwd(B=0) == 1 and fwd(mq=0) == 1 and fwd(tk=0) == 1
    assert fwd(d=80) == 2
    rc = lib.fa_forward_varlen(ptr, ptr, ptr, ptr, ptr, ptr, ptr, 2, 3, 100, 120, 150, 200, 64, 1, 1, 0.125, 1.5, 0,
                               0, None)
    assert rc == 1  # bad dropout probability
    ws = lib.fa_backward_varlen_workspace_size
    assert ws(150, 3, 96) == ((150 * 3 * 4 + 255) // 256) * 256 + 150 * 3 * 96 * 4
    assert ws(0, 3, 64) == 0 and ws(10, 3, 80) == 0
    rc = lib.fa_backward_varlen(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 2, 3, 100, 120, 150, 200, 64,
                                1, 1, 0.125, 0.0, 0, 0, ptr, 16, None)
    assert rc == 5  # workspace too small


def test_head_dim_256_has_no_block_mask(lib):
    ptr = 1 << 20
    assert lib.fa_backward_workspace_size(1, 1, 64, 256) == 256 + 64 * 256 * 4
    rc = lib.fa_forward_blocksparse(ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 1, 64, 256, 1, 0, 0.0625, None)
    assert rc == 2
    rc = lib.fa_backward_blocksparse(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, 1, 64, 256, 1, 0,
                                     0.0625, ptr, 1 << 30, None)
    assert rc == 2


def test_grouped_query_decode_validation(lib):
    """Query heads not a multiple of the K / V heads are rejected before any
    launch; the workspace of grouped decoding is that of plain decoding over
    the K / V heads with their query heads' rows stacked."""
    ptr = 1 << 20
    assert lib.fa_decode_gqa_workspace_size(1, 8, 3, 1, 1000, 128, 0) == 0
    assert lib.fa_decode_gqa_workspace_size(1, 8, 0, 1, 1000, 128, 0) == 0
    for splits in (0, 5):
        assert lib.fa_decode_gqa_workspace_size(2, 8, 2, 3, 1000, 128, splits) == \
            lib.fa_decode_workspace_size(2, 2, 12, 1000, 128, splits)
    assert lib.fa_decode_gqa_workspace_size(1, 4, 4, 2, 300, 64, 0) == lib.fa_decode_workspace_size(1, 4, 2, 300, 64, 0)
    rc = lib.fa_forward_decode_gqa(ptr, ptr, ptr, ptr, ptr, 1, 8, 3, 1, 1000, 128, 1, 1, 0.125, 0, ptr, 1 << 30, None)
    assert rc == 1
    rc = lib.fa_forward_decode_gqa(ptr, ptr, ptr, ptr, ptr, 1, 8, 2, 10, 5, 128, 1, 1, 0.125, 0, ptr, 1 << 30, None)
    assert rc == 1  # causal with more queries than keys

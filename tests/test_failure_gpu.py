"""Failure detection without a GPU fault: a pipeline wait that can never
complete (an mbarrier nothing arrives at) gives up after its bounded time,
latches FA_ERR_TIMEOUT in the device status word, and leaves the context
usable for the next call."""
import time

import pytest
import torch

import exact_io_aware_forward_gb300 as fa
from exact_io_aware_forward_gb300.synth import attention_inputs

pytestmark = pytest.mark.gpu


def test_stuck_wait_is_reported_and_the_context_survives():
    fa.fa_device_status()  # start from a clear status word
    t0 = time.perf_counter()
    fa.fa_selftest_wait_timeout()
    with pytest.raises(fa.FAError) as e:
        fa.fa_device_status()
    waited = time.perf_counter() - t0
    assert e.value.code == 4, e.value
    assert 1.0 < waited < 30.0, waited
    fa.fa_device_status()  # the report cleared the word
    q, k, v, _ = (x.to("cuda:0") if x is not None else None for x in attention_inputs(1, 2, 256, 64, "bf16", seed=1))
    o, lse = fa.forward(q, k, v, causal=True)
    fa.fa_device_status()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()

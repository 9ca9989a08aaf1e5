"""Failure detection on the GPU without a fault: a bounded in-kernel wait that nothing
completes gives up after its limit, reports ATTN_ERR_DEVICE_TIMEOUT through the device status
word, and leaves the CUDA context usable for the next call."""
import time

import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import masks
from synth import Workload

from helpers import check_forward, head_inputs, oracle_forward, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    assert ea.attn_device_status() == ea.ATTN_OK
    t0 = time.perf_counter()
    ea.attn_selftest_wait_timeout()
    with pytest.raises(ea.AttnError) as err:
        ea.attn_device_status()
    elapsed = time.perf_counter() - t0
    assert err.value.code == ea.ATTN_ERR_DEVICE_TIMEOUT
    assert "0x3f" in ea.attn_last_error()
    assert 1.5 < elapsed < 30.0
    # the word was cleared and the context still computes correct attention
    assert ea.attn_device_status() == ea.ATTN_OK
    wl = Workload("after_timeout", 12, 1, 2, 300, 64, "bf16", "causal", 0.125)
    inp = head_inputs(wl)
    dev = {t: to_dev(inp[t], "bf16") for t in inp}
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal")
    assert ea.attn_device_status() == ea.ATTN_OK
    Y, L = oracle_forward(inp, wl, masks.causal(wl.n))
    check_forward(o, lse, Y, L, "bf16", "after timeout")

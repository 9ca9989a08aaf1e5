"""Pipeline-depth invariance: every kernel gives bit-identical outputs with its shared-memory
rings capped at 1, 2, 3 and 4 stages (attn_debug_set_ring_stages) and at the default depth.

The ring depth only decides when a tile is loaded and which stage (and mbarrier phase parity)
it uses; the arithmetic and its order are the same.  The capped kernels are the instantiations
for bf16, d = 128, key block 128 without dropout, and the FP8 forward with d = 128 (the same
source as every other instantiation, with the stage counts read at launch).  A mistake in the stage/phase bookkeeping
(a wrong parity, a stage released early) either hangs a bounded wait (reported as a device
timeout) or feeds a product a stale tile, which changes bits.  Rings whose schedule needs two
stages (the backward's query-block ring and the dQ kernel's key ring) keep two at cap 1.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from synth import Workload, pack_bitmap, random_allowed

from helpers import head_inputs, to_dev

pytestmark = pytest.mark.gpu

CAPS = (1, 2, 3, 4)


@pytest.fixture(autouse=True)
def _reset_depth():
    ea.load()
    ea.attn_debug_set_ring_stages(0)
    yield
    ea.attn_debug_set_ring_stages(0)


def _bits(mask, n, seed=3):
    if mask != "bitmap":
        return None
    return torch.from_numpy(pack_bitmap(random_allowed(n, seed, keep=0.4)).view(np.int32)).cuda()


def _run_all(dev, c, mask, bits, kvb, drop):
    v, g = dev["v"], dev["do"]
    o, lse = ea.attn_fwd(dev["q"], dev["k"], v, c, mask=mask, mask_bits=bits, kv_block=kvb,
                         dropout_p=drop, seed=99)
    grads = ea.attn_bwd(dev["q"], dev["k"], v, o, lse, g, c, mask=mask, mask_bits=bits,
                        kv_block=kvb, dropout_p=drop, seed=99)
    assert ea.attn_device_status() in (ea.ATTN_OK, ea.ATTN_WARN_EMPTY_ROW)
    return (o, lse) + tuple(grads)


@pytest.mark.parametrize("mask,n,kvb,H", [
    ("none", 700, 128, 3), ("causal", 1100, 0, 3), ("bitmap", 513, 128, 3), ("causal", 4096, 0, 3),
    ("none", 128, 0, 3), ("bitmap", 1, 128, 3),
    # enough heads that the forward keeps two query tiles per CTA (grid over half the SMs)
    ("causal", 2048, 0, 10),
])
def test_outputs_do_not_depend_on_ring_depth(mask, n, kvb, H):
    d = 128
    wl = Workload("ring", 17, 1, H, n, d, "bf16", mask, d ** -0.5)
    inp = head_inputs(wl)
    dev = {t: to_dev(inp[t], "bf16") for t in inp}
    bits = _bits(mask, n)
    ref = _run_all(dev, wl.c, mask, bits, kvb, 0.0)
    for cap in CAPS:
        ea.attn_debug_set_ring_stages(cap)
        got = _run_all(dev, wl.c, mask, bits, kvb, 0.0)
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), got, ref):
            assert torch.equal(a, b), f"cap {cap}: {name} differs"


def test_other_calls_are_refused_while_a_cap_is_set():
    wl = Workload("ring_other", 18, 1, 1, 256, 64, "bf16", "none", 0.125)
    inp = head_inputs(wl)
    dev = {t: to_dev(inp[t], "bf16") for t in inp}
    ea.attn_debug_set_ring_stages(2)
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c)
    assert e.value.code == ea.ATTN_ERR_UNSUPPORTED
    ea.attn_debug_set_ring_stages(0)
    ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c)  # the default depth serves every shape
    assert ea.attn_device_status() == ea.ATTN_OK


def test_fp8_forward_does_not_depend_on_ring_depth():
    B, H, n, d = 1, 2, 640, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    xs = [torch.randn((B, H, n, d), device="cuda", generator=g) for _ in range(3)]
    q8, k8, v8 = (x.to(torch.float8_e4m3fn) for x in xs)
    vt8 = v8.transpose(2, 3).contiguous()
    ref = ea.attn_fwd_fp8(q8, k8, vt8, d ** -0.5, 1.0, 1.0, 1.0, mask="causal")
    for cap in CAPS:
        ea.attn_debug_set_ring_stages(cap)
        got = ea.attn_fwd_fp8(q8, k8, vt8, d ** -0.5, 1.0, 1.0, 1.0, mask="causal")
        assert ea.attn_device_status() == ea.ATTN_OK
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), f"cap {cap}"

"""GPU vs oracle parity on small problems that span several tiles and ragged tails.

Covers every dtype (float32 CUDA-core path, fp16 / bf16 tensor-core path), head dimension,
mask kind and key-block size, forward and backward, through the C ABI.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import masks
from synth import Workload, pack_bitmap, random_allowed

from helpers import (check_forward, check_grads, head_inputs, oracle_backward,
                     oracle_forward, to_dev)

pytestmark = pytest.mark.gpu

SHAPES = [(1, 2, 77, 32), (2, 1, 300, 64), (1, 1, 513, 128), (1, 1, 1, 0), (1, 2, 256, 64)]


def _cases():
    out = []
    for dtype in ("f32", "f16", "bf16"):
        for d in (16, 32, 64, 128):
            for mask in ("none", "causal", "bitmap"):
                for (B, H, n, kvb) in SHAPES:
                    out.append((dtype, d, mask, B, H, n, kvb))
    return out


def _setup(dtype, d, mask, B, H, n, kvb, seed=11):
    wl = Workload(f"small_{dtype}_{d}_{mask}_{n}", seed, B, H, n, d, dtype, mask,
                  1.0 / np.sqrt(d), kv_block=kvb)
    inp = head_inputs(wl)
    if mask == "bitmap":
        allowed = random_allowed(n, seed + n, keep=0.35)
        words = pack_bitmap(allowed)
        mk = masks.bitmap(words, n)
        bits = torch.from_numpy(words.view(np.int32)).cuda()
    else:
        mk, bits = masks.for_kind(mask, n), None
    dev = {t: to_dev(inp[t], dtype) for t in inp}
    return wl, inp, mk, bits, dev


@pytest.mark.parametrize("dtype,d,mask,B,H,n,kvb", _cases())
def test_forward_small(dtype, d, mask, B, H, n, kvb):
    ea.load()
    wl, inp, mk, bits, dev = _setup(dtype, d, mask, B, H, n, kvb)
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask=mask, mask_bits=bits,
                         kv_block=kvb)
    assert ea.attn_device_status() == ea.ATTN_OK
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, dtype, wl.name)


@pytest.mark.parametrize("dtype,d,mask,B,H,n,kvb", _cases())
def test_backward_small(dtype, d, mask, B, H, n, kvb):
    ea.load()
    wl, inp, mk, bits, dev = _setup(dtype, d, mask, B, H, n, kvb)
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask=mask, mask_bits=bits,
                         kv_block=kvb)
    dq, dk, dv = ea.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], wl.c, mask=mask,
                             mask_bits=bits, kv_block=kvb)
    assert ea.attn_device_status() == ea.ATTN_OK
    refs = oracle_backward(inp, wl, mk)
    check_grads((dq, dk, dv), refs, dtype, wl.name)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("mask", ["none", "causal", "bitmap"])
@pytest.mark.parametrize("kvb", [32, 64, 128])
def test_mask_membership_exact(dtype, mask, kvb):
    """c = 0 makes every allowed key weigh the same: LSE_i = ln |A_i| and O_i is the mean of
    V over A_i.  V encodes each key's index in binary, so O recovers, per row, the exact
    number of allowed keys with each index bit set: a fingerprint of the allowed set."""
    # O is rounded to the output type; the recovered per-bit counts stay exact while
    # count * 2^-(mantissa bits + 1) < 1/2, so bf16 runs use fewer keys per row.
    n, d = (250 if dtype == "bf16" else 600), 16
    wl = Workload("membership", 3, 1, 1, n, d, dtype, mask, 0.0, kv_block=kvb)
    inp = head_inputs(wl)
    j = np.arange(n)
    enc = ((j[:, None] >> np.arange(d)[None, :]) & 1).astype(np.float32)
    inp["v"][0, 0] = enc
    if mask == "bitmap":
        allowed = random_allowed(n, 99, keep=0.2)
        words = pack_bitmap(allowed)
        mk, bits = masks.bitmap(words, n), torch.from_numpy(words.view(np.int32)).cuda()
    else:
        mk, bits = masks.for_kind(mask, n), None
    dev = {t: to_dev(inp[t], dtype) for t in inp}
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], 0.0, mask=mask, mask_bits=bits,
                         kv_block=kvb)
    assert ea.attn_device_status() == ea.ATTN_OK
    a = mk(0, np.arange(n))
    count = a.sum(axis=1)
    lse = lse[0, 0].double().cpu().numpy()
    assert np.max(np.abs(lse - np.log(count))) <= 1e-5
    per_bit = np.rint(o[0, 0].double().cpu().numpy() * count[:, None])
    want = a.astype(np.int64) @ enc.astype(np.int64)
    assert np.array_equal(per_bit.astype(np.int64), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_rows_reading(dtype):
    """A row with no allowed key: O = 0, LSE = -inf, no gradient, status flag raised."""
    n, d = 200, 64
    wl = Workload("empty", 4, 1, 1, n, d, dtype, "bitmap", 0.125)
    inp = head_inputs(wl)
    allowed = random_allowed(n, 5, keep=0.3)
    allowed[[0, 130, 199]] = False
    allowed[:, 140:] = False
    words = pack_bitmap(allowed)
    mk, bits = masks.bitmap(words, n), torch.from_numpy(words.view(np.int32)).cuda()
    dev = {t: to_dev(inp[t], dtype) for t in inp}
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="bitmap", mask_bits=bits)
    assert ea.attn_device_status() == ea.ATTN_WARN_EMPTY_ROW
    dq, dk, dv = ea.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], wl.c,
                             mask="bitmap", mask_bits=bits)
    ea.attn_device_status()
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, dtype, "empty rows")
    assert torch.all(o[0, 0, [0, 130, 199]] == 0)
    refs = oracle_backward(inp, wl, mk)
    check_grads((dq, dk, dv), refs, dtype, "empty rows")
    assert torch.all(dk[0, 0, 140:] == 0) and torch.all(dv[0, 0, 140:] == 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_key_block_sizes_agree(dtype):
    """b in {32, 64, 128}: the same allowed sets and O within tolerance of each other."""
    n, d = 700, 64
    wl = Workload("kvb", 8, 1, 2, n, d, dtype, "causal", 0.125)
    inp = head_inputs(wl)
    dev = {t: to_dev(inp[t], dtype) for t in inp}
    outs = [ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal", kv_block=b)
            for b in (32, 64, 128)]
    Y, L = oracle_forward(inp, wl, masks.causal(n))
    for o, lse in outs:
        check_forward(o, lse, Y, L, dtype, "kv_block")
    a = outs[0][0].double()
    for o, _ in outs[1:]:
        assert torch.all((o.double() - a).abs() <= 2 * (2e-2 + 2e-2 * a.abs()))


def test_autograd_wrapper_matches_abi():
    n, d = 257, 64
    wl = Workload("autograd", 9, 1, 2, n, d, "bf16", "causal", 0.125)
    inp = head_inputs(wl)
    dev = {t: to_dev(inp[t], "bf16") for t in inp}
    q, k, v = (dev[t].clone().requires_grad_() for t in ("q", "k", "v"))
    y = ea.attention(q, k, v, wl.c, mask="causal")
    y.backward(dev["do"])
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal")
    dq, dk, dv = ea.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], wl.c, mask="causal")
    assert torch.equal(y, o)
    assert torch.equal(q.grad, dq) and torch.equal(k.grad, dk) and torch.equal(v.grad, dv)

"""Bitmap masks over more than 32 blocks of 128, with whole blocks empty between taken ones.

The kernels compact a bitmap's taken blocks into a step list 32 blocks at a time (the
forward per query pair over key blocks, the dK/dV kernel per key tile over query blocks), and
the small parity shapes reach fewer than 32 blocks.  Here n = 40 blocks + a ragged tail, and
query block i sees key block j only when (i + 2 j) mod 3 != 0 (elementwise a random third of
those pairs, the diagonal always), so every row's and every key's run of blocks has gaps
spread over both rounds of the compaction.  Forward and backward are compared with the oracle
on whole heads.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import masks
from synth import Workload, pack_bitmap, random_allowed

from helpers import check_forward, check_grads, head_inputs, oracle_backward, oracle_forward, to_dev

pytestmark = pytest.mark.gpu

N = 40 * 128 + 77


def _allowed(n, seed):
    blk = np.arange(n) // 128
    taken = (blk[:, None] + 2 * blk[None, :]) % 3 != 0
    a = random_allowed(n, seed, keep=0.35) & taken
    a[np.arange(n), np.arange(n)] = True
    return a


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("kvb", [128, 64])
def test_bitmap_over_forty_blocks(dtype, kvb):
    ea.load()
    wl = Workload(f"bitmap_many_{dtype}_{kvb}", 61, 1, 1, N, 64, dtype, "bitmap", 0.125,
                  kv_block=kvb)
    inp = head_inputs(wl)
    allowed = _allowed(N, 62)
    words = pack_bitmap(allowed)
    mk = masks.bitmap(words, N)
    bits = torch.from_numpy(words.view(np.int32)).cuda()
    dev = {t: to_dev(inp[t], dtype) for t in inp}
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="bitmap", mask_bits=bits,
                         kv_block=kvb)
    dq, dk, dv = ea.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], wl.c,
                             mask="bitmap", mask_bits=bits, kv_block=kvb)
    assert ea.attn_device_status() == ea.ATTN_OK
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, dtype, wl.name)
    check_grads((dq, dk, dv), oracle_backward(inp, wl, mk), dtype, wl.name)

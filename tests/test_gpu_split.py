"""Key-split forward and the merge of partial results, on the GPU, against the oracle.

attn_fwd_split cuts each row's key blocks into shares, summarises every share in its own CTA
and merges the shares (the merge rule of the stable summaries in "Exact tiled attention and
memory-aware differentiation").  The merged result must equal the oracle's dense forward
within the forward tolerances, for every mask, dtype, share count (including more shares than
key blocks, which leaves some shares empty) and key-block size.  attn_merge is checked on
its own against the oracle's merge of normalised parts, including empty parts and rows whose
parts are all empty.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import masks, tiled
from synth import Workload, draw_head, workload

from helpers import check_forward, head_inputs, mask_for, oracle_forward, to_dev

pytestmark = pytest.mark.gpu


def _run_split(wl, splits, kv_block=0):
    inp = head_inputs(wl)
    mk, bits, _ = mask_for(wl)
    dev = {t: to_dev(inp[t], wl.dtype) for t in ("q", "k", "v")}
    o, lse = ea.attn_fwd_split(dev["q"], dev["k"], dev["v"], wl.c, mask=wl.mask, mask_bits=bits,
                               kv_block=kv_block, num_splits=splits)
    status = ea.attn_device_status()
    return inp, mk, dev, bits, o, lse, status


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mask", ["none", "causal", "bitmap"])
@pytest.mark.parametrize("splits", [2, 5])
@pytest.mark.parametrize("d", [64, 128])
def test_split_forward_matches_oracle(dtype, mask, splits, d):
    wl = Workload("split", 41, 1, 2, 700, d, dtype, mask, d ** -0.5)
    inp, mk, dev, bits, o, lse, status = _run_split(wl, splits)
    assert status == ea.ATTN_OK
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, dtype, f"split {splits} {mask} {dtype} d={d}")
    # and the unsplit forward on the same inputs agrees within the same bounds
    o1, l1 = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask=mask, mask_bits=bits)
    check_forward(o, lse, o1.double().cpu().numpy(), l1.double().cpu().numpy(), dtype, "vs attn_fwd")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("kv_block", [32, 64, 128])
def test_split_bitmap_key_blocks(dtype, kv_block):
    wl = Workload("split_bitmap", 42, 2, 1, 523, 64, dtype, "bitmap", 0.125)
    inp, mk, _, _, o, lse, status = _run_split(wl, 3, kv_block)
    assert status == ea.ATTN_OK
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, dtype, f"bitmap b={kv_block}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n,splits", [(1, 4), (130, 7), (300, 32), (257, 3)])
def test_split_edges(dtype, n, splits):
    """More shares than key blocks (empty shares), a single row, ragged tiles."""
    wl = Workload("split_edge", 43, 1, 3, n, 64, dtype, "causal", 0.3)
    inp, mk, _, _, o, lse, status = _run_split(wl, splits)
    assert status == ea.ATTN_OK
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, dtype, f"n={n} splits={splits}")


def test_split_library_choice_fills_the_gpu():
    wl = Workload("split_auto", 44, 1, 1, 2048, 64, "bf16", "causal", 0.125)
    count = ea.attn_fwd_split_count(torch.bfloat16, wl.B, wl.H, wl.n, wl.d)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert count > 1 and count * 8 >= min(sms, 8 * 16)  # 8 CTAs per share, one share per block
    inp, mk, _, _, o, lse, status = _run_split(wl, 0)
    assert status == ea.ATTN_OK
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, "bf16", "library choice")


def test_split_empty_rows_flagged_once_merged():
    """A row with no allowed key anywhere is an empty row after the merge (O = 0, LSE = -inf,
    flag); a row that is empty only within some shares is not."""
    n = 300
    allowed = np.zeros((n, n), bool)
    allowed[np.arange(n), np.arange(n)] = True
    allowed[7] = False  # row 7: nothing allowed
    wl = Workload("split_empty", 45, 1, 1, n, 64, "bf16", "bitmap", 0.125)
    inp = head_inputs(wl)
    mk, bits, _ = mask_for(wl, allowed)
    dev = {t: to_dev(inp[t], "bf16") for t in ("q", "k", "v")}
    o, lse = ea.attn_fwd_split(dev["q"], dev["k"], dev["v"], wl.c, mask="bitmap", mask_bits=bits,
                               num_splits=3)
    assert ea.attn_device_status() == ea.ATTN_WARN_EMPTY_ROW
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, "bf16", "empty row")
    assert float(lse[0, 0, 7]) == -math.inf and bool((o[0, 0, 7] == 0).all())


@pytest.mark.parametrize("name", ["overflow_f16_d16", "overflow_f16_d64_hot"])
def test_split_overflow_workloads_full_size(name):
    """The few-head fp16 workloads at full size through the library's split choice."""
    wl = workload(name)
    dev = {}
    for t in ("q", "k", "v"):
        x = torch.empty((wl.B, wl.H, wl.n, wl.d), dtype=torch.float16, device="cuda")
        for bh in range(wl.heads):
            x[bh // wl.H, bh % wl.H] = to_dev(draw_head(wl, t, bh), "f16")
        dev[t] = x
    o, lse = ea.attn_fwd_split(dev["q"], dev["k"], dev["v"], wl.c, mask="causal")
    assert ea.attn_device_status() == ea.ATTN_OK
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, wl.n // 2, wl.n - 1],
                                     rng.choice(wl.n, 256, replace=False)]))
    from oracle import attention as ref
    for bh in range(wl.heads):
        q = draw_head(wl, "q", bh)[rows]
        y, l, _, _ = ref.forward_rows(q, draw_head(wl, "k", bh), draw_head(wl, "v", bh), wl.c,
                                      masks.causal(wl.n)(bh, rows))
        idx = torch.from_numpy(rows).cuda()
        check_forward(o[0, bh].index_select(0, idx), lse[0, bh].index_select(0, idx), y, l, "f16",
                      f"{name} head {bh}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_merge_matches_oracle(dtype):
    rng = np.random.default_rng(7)
    parts, rows, d = 4, 37, 64
    o_parts = rng.normal(size=(parts, rows, d)).astype(np.float32)
    lse_parts = (rng.normal(size=(parts, rows)) * 6).astype(np.float32)
    lse_parts[rng.random((parts, rows)) < 0.3] = -np.inf  # empty parts
    lse_parts[:, 5] = -np.inf  # a row with every part empty
    lse_parts[0, 9], lse_parts[1:, 9] = 1.5, -np.inf  # a row with one nonempty part
    o, lse = ea.attn_merge(torch.from_numpy(o_parts).cuda(), torch.from_numpy(lse_parts).cuda(),
                           dtype={"f32": torch.float32, "f16": torch.float16,
                                  "bf16": torch.bfloat16}[dtype])
    assert ea.attn_device_status() == ea.ATTN_WARN_EMPTY_ROW  # row 5
    want_o = np.zeros((rows, d))
    want_l = np.zeros(rows)
    for r in range(rows):
        want_o[r], want_l[r] = tiled.merge_normalised(
            [(o_parts[g, r].astype(np.float64), float(lse_parts[g, r])) for g in range(parts)])
    got_o = o.double().cpu().numpy()
    got_l = lse.double().cpu().numpy()
    assert got_l[5] == -np.inf and np.all(got_o[5] == 0)
    fin = np.isfinite(want_l)
    assert np.all(np.isfinite(got_l[fin]))
    assert np.max(np.abs(got_l[fin] - want_l[fin])) <= 1e-5
    tol = 1e-5 if dtype == "f32" else 1e-2
    assert np.all(np.abs(got_o - want_o) <= tol * (1 + np.abs(want_o)))
    if dtype == "f32":  # one nonempty part: passed through unchanged
        assert np.max(np.abs(got_o[9] - o_parts[0, 9])) <= 1e-6


@pytest.mark.parametrize("splits", [None, 2])
def test_tile_with_no_allowed_key(splits):
    """A whole 128-row tile whose rows allow no key (bitmap) takes no step at all; its rows are
    still written as empty rows (O = 0, LSE = -inf, flag), through attn_fwd and the split path."""
    n = 300
    allowed = np.zeros((n, n), bool)
    allowed[np.arange(n), np.arange(n)] = True
    allowed[128:256] = False
    wl = Workload("empty_tile", 46, 1, 1, n, 64, "bf16", "bitmap", 0.125)
    inp = head_inputs(wl)
    mk, bits, _ = mask_for(wl, allowed)
    dev = {t: to_dev(inp[t], "bf16") for t in ("q", "k", "v")}
    if splits is None:
        o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="bitmap", mask_bits=bits)
    else:
        o, lse = ea.attn_fwd_split(dev["q"], dev["k"], dev["v"], wl.c, mask="bitmap",
                                   mask_bits=bits, num_splits=splits)
    assert ea.attn_device_status() == ea.ATTN_WARN_EMPTY_ROW
    Y, L = oracle_forward(inp, wl, mk)
    check_forward(o, lse, Y, L, "bf16", f"empty tile, splits={splits}")
    assert bool((lse[0, 0, 128:256] == -math.inf).all()) and bool((o[0, 0, 128:256] == 0).all())

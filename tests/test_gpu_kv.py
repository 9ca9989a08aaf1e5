"""Forward over a key/value cache (n_q query rows against n_kv keys), on the GPU, vs the oracle.

attn_fwd_kv places the queries at the end of the sequence (under the causal mask query i sees
keys j <= i + n_kv - n_q) and cuts the keys into shares merged by the rule of the stable
summaries.  Checked here: every dtype and mask against the oracle's dense forward on the same
rectangle, more query rows than keys (empty rows), the reduction to attn_fwd at n_q = n_kv, the
cache identity (the last rows of square causal attention), and a full-size decoding shape.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import attention as ref
from oracle import masks
from synth import Workload, draw_head, pack_bitmap

from helpers import check_forward, to_dev

pytestmark = pytest.mark.gpu


def _inputs(wl, nq, nk):
    q = np.stack([draw_head(wl, "q", bh, nq) for bh in range(wl.heads)])
    k = np.stack([draw_head(wl, "k", bh, nk) for bh in range(wl.heads)])
    v = np.stack([draw_head(wl, "v", bh, nk) for bh in range(wl.heads)])
    shape = lambda x: x.reshape(wl.B, wl.H, *x.shape[1:])
    return shape(q), shape(k), shape(v)


def _mask(kind, nq, nk, seed=0):
    if kind == "none":
        return masks.none(nk), None
    if kind == "causal":
        return masks.causal_rect(nq, nk), None
    rng = np.random.default_rng(seed)
    allowed = rng.random((nq, nk)) < 0.3
    allowed[np.arange(nq), rng.integers(0, nk, nq)] = True
    words = pack_bitmap(allowed)
    return masks.bitmap(words, nk), torch.from_numpy(words.view(np.int32)).cuda()


def _oracle(q, k, v, c, mk):
    B, H, nq, d = q.shape
    Y = np.zeros((B, H, nq, d))
    L = np.zeros((B, H, nq))
    for bh in range(B * H):
        b, h = divmod(bh, H)
        Y[b, h], L[b, h], _, _ = ref.forward_rows(q[b, h], k[b, h], v[b, h], c,
                                                  mk(bh, np.arange(nq)))
    return Y, L


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mask", ["none", "causal", "bitmap"])
@pytest.mark.parametrize("nq,nk", [(1, 777), (3, 1000), (130, 300), (300, 130), (256, 2048)])
@pytest.mark.parametrize("splits", [0, 1, 4])
def test_kv_forward_matches_oracle(dtype, mask, nq, nk, splits):
    d = 64
    wl = Workload("kv", 61, 1, 2, max(nq, nk), d, dtype, mask, d ** -0.5)
    q, k, v = _inputs(wl, nq, nk)
    mk, bits = _mask(mask, nq, nk, 7)
    dq, dk, dv = (to_dev(x, dtype) for x in (q, k, v))
    o, lse = ea.attn_fwd_kv(dq, dk, dv, wl.c, mask=mask, mask_bits=bits, num_splits=splits)
    status = ea.attn_device_status()
    Y, L = _oracle(q, k, v, wl.c, mk)
    empty = ~np.isfinite(L)
    assert status == (ea.ATTN_WARN_EMPTY_ROW if empty.any() else ea.ATTN_OK)
    check_forward(o, lse, Y, L, dtype, f"kv {nq}x{nk} {mask} {dtype} splits={splits}")


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_kv_equal_lengths_is_attn_fwd(mask):
    wl = Workload("kv_sq", 62, 2, 2, 400, 128, "bf16", mask, 128 ** -0.5)
    q, k, v = (to_dev(x, "bf16") for x in _inputs(wl, 400, 400))
    o1, l1 = ea.attn_fwd(q, k, v, wl.c, mask=mask)
    o2, l2 = ea.attn_fwd_kv(q, k, v, wl.c, mask=mask, num_splits=1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kv_cache_is_the_tail_of_causal_attention(dtype):
    n, m = 1000, 37
    wl = Workload("kv_tail", 63, 1, 3, n, 64, dtype, "causal", 0.125)
    q, k, v = (to_dev(x, dtype) for x in _inputs(wl, n, n))
    o, lse = ea.attn_fwd(q, k, v, wl.c, mask="causal")
    ot, lt = ea.attn_fwd_kv(q[:, :, n - m:].contiguous(), k, v, wl.c, mask="causal")
    check_forward(ot, lt, o[:, :, n - m:].double().cpu().numpy(),
                  lse[:, :, n - m:].double().cpu().numpy(), dtype, "cache tail")


def test_decoding_shape_full_size():
    """One query per head against a 32768-key cache, 8 x 32 heads, d = 128, bf16: the library's
    share choice; sampled heads against the oracle, every output finite."""
    B, H, nk, d = 8, 32, 32768, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    q = torch.randn((B, H, 1, d), device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, nk, d), device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, nk, d), device="cuda", generator=g).to(torch.bfloat16)
    c = d ** -0.5
    assert ea.attn_fwd_kv_split_count(torch.bfloat16, B, H, 1, nk, d) > 1
    o, lse = ea.attn_fwd_kv(q, k, v, c, mask="causal")
    assert ea.attn_device_status() == ea.ATTN_OK
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    for bh in (0, 77, 255):
        b, h = divmod(bh, H)
        qq, kk, vv = (x[b, h].double().cpu().numpy() for x in (q, k, v))
        y, l, _, _ = ref.forward_rows(qq, kk, vv, c, np.ones((1, nk), bool))
        check_forward(o[b, h], lse[b, h], y, l, "bf16", f"decode head {bh}")

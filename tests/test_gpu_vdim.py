"""Values of their own width (v != d), on the GPU, against the oracle.

"Exact tiled attention and memory-aware differentiation" states the problem with Q, K in
R^{n x d} and V in R^{n x v}: the scores and their gradients live in the d-wide space, O, dO
and dV in the v-wide one.  The library runs (d, v) = (64, 128) and (128, 64) in every dtype;
the oracle's dense definition takes any widths (its reverse procedure is pinned against finite
differences with v != d on the CPU).
"""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import attention as ref
from oracle import dropout as odrop
from synth import Workload, draw_head

from helpers import check_forward, mask_for, rel_frob_per_head, to_dev, tol_grad

pytestmark = pytest.mark.gpu


def _inputs(B, H, n, d, vw, dtype, mask, seed):
    """q, k of width d and v, do of width vw, drawn head by head (dtype-rounded)."""
    wq = Workload("vdim", seed, B, H, n, d, dtype, mask, d ** -0.5)
    wv = Workload("vdim_v", seed + 1, B, H, n, vw, dtype, mask, d ** -0.5)
    x = {}
    for t, wl in (("q", wq), ("k", wq), ("v", wv), ("do", wv)):
        x[t] = np.stack([draw_head(wl, t, bh) for bh in range(B * H)]).reshape(B, H, n, wl.d)
    return wq, x


def _run(x, wl, dtype, mask, bits, kv_block=0, dropout_p=0.0, seed=0):
    dev = {t: to_dev(x[t], dtype) for t in x}
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask=mask, mask_bits=bits,
                         kv_block=kv_block, dropout_p=dropout_p, seed=seed)
    dq, dk, dv = ea.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], wl.c, mask=mask,
                             mask_bits=bits, kv_block=kv_block, dropout_p=dropout_p, seed=seed)
    status = ea.attn_device_status()
    return status, o, lse, (dq, dk, dv)


def _check_grads(got, want, dtype, what):
    for name, g, w in zip(("dQ", "dK", "dV"), got, want):
        assert tuple(g.shape) == w.shape, f"{what} {name} shape"
        assert torch.isfinite(g).all(), f"{what} {name} not finite"
        err = rel_frob_per_head(g, w)
        assert err.max() <= tol_grad(dtype), f"{what} {name}: rel Frobenius {err.max():.3e}"


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("d,vw", [(64, 128), (128, 64)])
@pytest.mark.parametrize("mask", ["none", "causal", "bitmap"])
def test_forward_and_backward_match_the_oracle(dtype, d, vw, mask):
    B, H, n = 1, 2, 333  # three query tiles, ragged tail
    wl, x = _inputs(B, H, n, d, vw, dtype, mask, 91)
    mk, bits, _ = mask_for(wl)
    status, o, lse, grads = _run(x, wl, dtype, mask, bits)
    assert status == ea.ATTN_OK
    assert tuple(o.shape) == (B, H, n, vw)
    Y, L = ref.forward(x["q"], x["k"], x["v"], wl.c, mk)
    want = ref.backward(x["q"], x["k"], x["v"], wl.c, mk, x["do"])
    check_forward(o, lse, Y, L, dtype, f"v={vw} d={d} {mask} {dtype}")
    _check_grads(grads, want, dtype, f"v={vw} d={d} {mask} {dtype}")


@pytest.mark.parametrize("kv_block", [32, 64, 128])
@pytest.mark.parametrize("d,vw", [(64, 128), (128, 64)])
def test_key_blocks_and_dropout(kv_block, d, vw):
    B, H, n, p = 1, 2, 300, 0.2
    wl, x = _inputs(B, H, n, d, vw, "bf16", "causal", 92)
    mk, bits, _ = mask_for(wl)
    p32 = float(np.float32(p))
    status, o, lse, grads = _run(x, wl, "bf16", "causal", bits, kv_block, p32, 1234)
    assert status == ea.ATTN_OK
    rows = np.arange(n)
    Y = np.zeros((B, H, n, vw))
    L = np.zeros((B, H, n))
    want = [np.zeros((B, H, n, d)), np.zeros((B, H, n, d)), np.zeros((B, H, n, vw))]
    for bh in range(B * H):
        b, h = divmod(bh, H)
        keep = odrop.keep_mask(1234, bh, rows, n, p32)
        a = mk(bh, rows)
        Y[b, h], L[b, h] = odrop.forward_rows(x["q"][b, h], x["k"][b, h], x["v"][b, h], wl.c, a,
                                              keep, p32)
        for t, g in zip(want, odrop.backward_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], wl.c,
                                                  a, keep, p32, x["do"][b, h])):
            t[b, h] = g
    check_forward(o, lse, Y, L, "bf16", f"dropout b={kv_block}")
    _check_grads(grads, want, "bf16", f"dropout b={kv_block}")


@pytest.mark.parametrize("n", [1, 129])
@pytest.mark.parametrize("d,vw", [(64, 128), (128, 64)])
def test_single_row_and_one_past_a_tile(n, d, vw):
    B, H = 1, 3
    wl, x = _inputs(B, H, n, d, vw, "bf16", "causal", 95)
    mk, bits, _ = mask_for(wl)
    status, o, lse, grads = _run(x, wl, "bf16", "causal", bits)
    assert status == ea.ATTN_OK
    Y, L = ref.forward(x["q"], x["k"], x["v"], wl.c, mk)
    want = ref.backward(x["q"], x["k"], x["v"], wl.c, mk, x["do"])
    check_forward(o, lse, Y, L, "bf16", f"n={n} v={vw}")
    _check_grads(grads, want, "bf16", f"n={n} v={vw}")


def test_several_tiles_and_heads():
    B, H, n, d, vw = 2, 2, 1024, 128, 64
    wl, x = _inputs(B, H, n, d, vw, "bf16", "none", 93)
    mk, bits, _ = mask_for(wl)
    status, o, lse, grads = _run(x, wl, "bf16", "none", bits)
    assert status == ea.ATTN_OK
    heads = [0, 3]
    Y, L = ref.forward(x["q"], x["k"], x["v"], wl.c, mk, heads=heads)
    want = ref.backward(x["q"], x["k"], x["v"], wl.c, mk, x["do"], heads=heads)
    for bh in heads:
        b, h = divmod(bh, H)
        check_forward(o[b, h], lse[b, h], Y[b, h], L[b, h], "bf16", f"head {bh}")
        for g, w in zip(grads, want):
            assert rel_frob_per_head(g[b, h][None], w[b, h][None]).max() <= tol_grad("bf16")


def test_autograd_wrapper():
    B, H, n, d, vw = 1, 2, 200, 64, 128
    wl, x = _inputs(B, H, n, d, vw, "bf16", "causal", 94)
    mk, _, _ = mask_for(wl)
    q, k, v = (to_dev(x[t], "bf16").requires_grad_() for t in ("q", "k", "v"))
    y = ea.attention(q, k, v, wl.c, mask="causal")
    assert tuple(y.shape) == (B, H, n, vw)
    y.backward(to_dev(x["do"], "bf16"))
    want = ref.backward(x["q"], x["k"], x["v"], wl.c, mk, x["do"])
    _check_grads((q.grad, k.grad, v.grad), want, "bf16", "autograd")


def test_unsupported_pairs_are_refused():
    q = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 1, 64, 32), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd(q, q, v, 0.1)
    assert e.value.code == ea.ATTN_ERR_UNSUPPORTED
    lib = ea.load()
    p = ea._ptr(q)
    assert lib.attn_fwd_vdim(2, 1, 1, 64, 64, 16, 0.1, p, p, p, 0, None, 0, 0, 0, 0.0, 0, p, p,
                             None) == ea.ATTN_ERR_UNSUPPORTED

"""Dropout with a replayed realised mask, on the GPU, against the oracle.

The mask is a pure function of (seed, head, query row, key) (Philox4x32-10, see
oracle/dropout.py), so it must match the oracle's bit for bit.  Two constructions read the
mask straight out of the outputs: with c = 0 every allowed probability of a row equals
1/|A_i|, so one-hot value rows make O_i show which keys row i kept, and one-hot upstream
gradients make dV show them for the backward.  The other tests compare O, LSE and the
gradients with the oracle's dropout forward and reverse pass on seeded inputs.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import dropout as odrop
from synth import Workload, pack_bitmap

from helpers import TORCH_DTYPE, check_forward, head_inputs, mask_for, rel_frob_per_head, to_dev, \
    tol_grad

pytestmark = pytest.mark.gpu

SEED = 0x5EED_1234_ABCD


def _window_bits(n, lo, width):
    allowed = np.zeros((n, n), bool)
    allowed[:, lo:lo + width] = True
    return allowed, torch.from_numpy(pack_bitmap(allowed).view(np.int32)).cuda()


@pytest.mark.parametrize("dtype,kvb", [("bf16", 128), ("bf16", 64), ("bf16", 32), ("f16", 0),
                                       ("f32", 0)])
@pytest.mark.parametrize("p", [0.3, 0.75])
def test_forward_mask_is_bit_exact(dtype, kvb, p):
    """c = 0 and a 128-key window J0.. per row: O[i, a] = keep(i, J0 + a) / (128 (1 - p')), p' the
    drop probability at the mask's 1/256 resolution."""
    B, H, n, d, j0 = 1, 3, 1000, 128, 640
    allowed, bits = _window_bits(n, j0, d)
    v = torch.zeros((B, H, n, d), dtype=TORCH_DTYPE[dtype], device="cuda")
    v[:, :, j0:j0 + d] = torch.eye(d, dtype=v.dtype, device="cuda")
    q = torch.randn((B, H, n, d), device="cuda").to(v.dtype)
    k = torch.randn((B, H, n, d), device="cuda").to(v.dtype)
    p32 = float(np.float32(p))
    o, lse = ea.attn_fwd(q, k, v, 0.0, mask="bitmap", mask_bits=bits, dropout_p=p32, seed=SEED,
                         kv_block=kvb)
    assert ea.attn_device_status() == ea.ATTN_OK
    got = (o.float().cpu().numpy() != 0)
    for bh in range(B * H):
        want = odrop.keep_mask(SEED, bh, np.arange(n), n, p32)[:, j0:j0 + d]
        assert np.array_equal(got[bh // H, bh % H], want), f"head {bh}"
    nz = o.float()[o != 0]
    pe = odrop.effective_p(p32)
    assert torch.allclose(nz, torch.full_like(nz, 1.0 / (d * (1.0 - pe))), rtol=1e-2)
    assert torch.allclose(lse, torch.full_like(lse, float(np.log(d))), atol=1e-5)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_mask_is_bit_exact(dtype):
    """c = 0, n = d = 128, dO_i = e_i: dV[j, a] = keep(a, j) / (128 (1 - p'))."""
    B, H, n, d, p = 1, 2, 128, 128, 0.4
    p32 = float(np.float32(p))
    dt = TORCH_DTYPE[dtype]
    q, k, v = (torch.randn((B, H, n, d), device="cuda").to(dt) for _ in range(3))
    do = torch.eye(n, dtype=dt, device="cuda").expand(B, H, n, d).contiguous()
    o, lse = ea.attn_fwd(q, k, v, 0.0, dropout_p=p32, seed=SEED)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, do, 0.0, dropout_p=p32, seed=SEED)
    assert ea.attn_device_status() == ea.ATTN_OK
    got = dv.float().cpu().numpy() != 0
    for bh in range(B * H):
        want = odrop.keep_mask(SEED, bh, np.arange(n), n, p32).T  # [key j, query a]
        assert np.array_equal(got[0, bh], want), f"head {bh}"
    assert float(dq.abs().max()) == 0.0 and float(dk.abs().max()) == 0.0  # c = 0


def _oracle(inp, wl, mk, p, seed):
    Y = np.zeros((wl.B, wl.H, wl.n, wl.d))
    L = np.zeros((wl.B, wl.H, wl.n))
    grads = [np.zeros((wl.B, wl.H, wl.n, wl.d)) for _ in range(3)]
    rows = np.arange(wl.n)
    for bh in range(wl.heads):
        b, h = divmod(bh, wl.H)
        a = mk(bh, rows)
        keep = odrop.keep_mask(seed, bh, rows, wl.n, p)
        q, k, v, g = (inp[t][b, h].astype(np.float64) for t in ("q", "k", "v", "do"))
        Y[b, h], L[b, h] = odrop.forward_rows(q, k, v, wl.c, a, keep, p)
        for t, x in zip(grads, odrop.backward_head(q, k, v, wl.c, a, keep, p, g)):
            t[b, h] = x
    return Y, L, grads


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("mask", ["none", "causal", "bitmap"])
@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout_matches_oracle(dtype, mask, p):
    d = 64 if dtype == "f32" else 128
    wl = Workload("dropout", 51, 1, 2, 333, d, dtype, mask, d ** -0.5)
    p32 = float(np.float32(p))
    inp = head_inputs(wl)
    mk, bits, _ = mask_for(wl)
    dev = {t: to_dev(inp[t], dtype) for t in inp}
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask=mask, mask_bits=bits,
                         dropout_p=p32, seed=SEED)
    dq, dk, dv = ea.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], wl.c, mask=mask,
                             mask_bits=bits, dropout_p=p32, seed=SEED)
    assert ea.attn_device_status() == ea.ATTN_OK
    Y, L, grads = _oracle(inp, wl, mk, p32, SEED)
    check_forward(o, lse, Y, L, dtype, f"dropout {p} {mask} {dtype}")
    for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), grads):
        assert torch.isfinite(got).all()
        err = rel_frob_per_head(got, want)
        assert err.max() <= tol_grad(dtype), f"{name} rel Frobenius {err.max():.3e}"


@pytest.mark.parametrize("kv_block", [32, 64])
def test_dropout_key_block_does_not_change_the_mask(kv_block):
    wl = Workload("dropout_b", 52, 1, 1, 300, 64, "bf16", "causal", 0.125)
    inp = head_inputs(wl)
    dev = {t: to_dev(inp[t], "bf16") for t in ("q", "k", "v")}
    o1, l1 = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal", dropout_p=0.25,
                         seed=7)
    o2, l2 = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal", kv_block=kv_block,
                         dropout_p=0.25, seed=7)
    check_forward(o2, l2, o1.double().cpu().numpy(), l1.double().cpu().numpy(), "bf16", "b")


def test_zero_probability_and_determinism():
    wl = Workload("dropout_det", 53, 2, 2, 257, 64, "bf16", "causal", 0.125)
    inp = head_inputs(wl)
    dev = {t: to_dev(inp[t], "bf16") for t in inp}
    o0, l0 = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal")
    oz, lz = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal", dropout_p=0.0, seed=3)
    assert torch.equal(o0, oz) and torch.equal(l0, lz)
    a1 = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal", dropout_p=0.2, seed=3)
    a2 = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal", dropout_p=0.2, seed=3)
    b1 = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal", dropout_p=0.2, seed=4)
    assert torch.equal(a1[0], a2[0]) and not torch.equal(a1[0], b1[0])
    assert torch.equal(a1[1], l0)  # LSE is that of the undropped scores
    lib = ea.load()
    rc = lib.attn_fwd_dropout(2, 1, 1, 16, 64, 0.1, ea._ptr(dev["q"]), ea._ptr(dev["k"]),
                              ea._ptr(dev["v"]), 0, None, 0, 0, 0, 1.0, 1, ea._ptr(oz),
                              ea._ptr(lz), None)
    assert rc == ea.ATTN_ERR_INVALID_ARG  # p_drop = 1 is refused
    rc = lib.attn_fwd_dropout(2, 1, 1, 16, 64, 0.1, ea._ptr(dev["q"]), ea._ptr(dev["k"]),
                              ea._ptr(dev["v"]), 0, None, 0, 0, 0, 0.999, 1, ea._ptr(oz),
                              ea._ptr(lz), None)
    assert rc == ea.ATTN_ERR_INVALID_ARG  # rounds to 1 at the mask's 1/256 resolution


def test_autograd_wrapper_with_dropout():
    wl = Workload("dropout_ag", 54, 1, 2, 200, 64, "bf16", "none", 0.125)
    inp = head_inputs(wl)
    q, k, v = (to_dev(inp[t], "bf16").requires_grad_() for t in ("q", "k", "v"))
    g = to_dev(inp["do"], "bf16")
    y = ea.attention(q, k, v, wl.c, dropout_p=0.3, seed=99)
    y.backward(g)
    mk, _, _ = mask_for(wl)
    Y, L, grads = _oracle(inp, wl, mk, float(np.float32(0.3)), 99)
    check_forward(y.detach(), torch.from_numpy(L), Y, L, "bf16", "autograd")
    for got, want in zip((q.grad, k.grad, v.grad), grads):
        assert rel_frob_per_head(got, want).max() <= tol_grad("bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_dq_kernel_mask_is_bit_exact(dtype):
    """The query-tile kernel's mask, read out of dQ: with the keys one-hot in a 128-key window,
    dQ[i, b] = c γ_{i, j0+b} is a single product, and a kept or dropped pair changes it by
    c P_ij dP_ij / (1 - p').  Every element must lie nearer the value its mask bit gives than the
    value the flipped bit would give (where the two differ by more than rounding)."""
    B, H, n, d, p = 1, 1, 300, 128, 0.4
    j0 = 128
    p32 = float(np.float32(p))
    pe = odrop.effective_p(p32)
    wl = Workload("dropout_dq", 55, B, H, n, d, dtype, "causal", d ** -0.5)
    inp = head_inputs(wl)
    kk = np.zeros((B, H, n, d), np.float32)
    kk[0, 0, j0:j0 + d] = np.eye(d, dtype=np.float32)
    inp["k"] = kk
    dev = {t: to_dev(inp[t], dtype) for t in inp}
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], wl.c, mask="causal", dropout_p=p32,
                         seed=SEED)
    dq, _, _ = ea.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], wl.c, mask="causal",
                           dropout_p=p32, seed=SEED)
    assert ea.attn_device_status() == ea.ATTN_OK
    rows = np.arange(n)
    a = np.tril(np.ones((n, n), bool))
    keep = odrop.keep_mask(SEED, 0, rows, n, p32)
    P, dPt, gamma = odrop.probabilities_and_gamma(*(inp[t][0, 0] for t in ("q", "k", "v")), wl.c,
                                                  a, keep, p32, inp["do"][0, 0])
    keys = np.arange(j0, j0 + d)
    want = wl.c * gamma[:, keys]
    flip = wl.c * (gamma + P * dPt / (1.0 - pe) * (1 - 2 * keep))[:, keys]
    got = dq[0, 0].double().cpu().numpy()
    sep = np.abs(want - flip) > 1e-2 * (np.abs(want) + np.abs(flip)) + 1e-6
    assert sep.sum() > 0.5 * a[:, keys].sum()
    nearer = np.abs(got - want) < np.abs(got - flip)
    bad = sep & ~nearer
    assert not bad.any(), f"mask bit wrong at {np.argwhere(bad)[:5].tolist()}"

"""Shared helpers of the GPU tests: seeded inputs to device tensors, oracle references and
the tolerance checks stated for this path.

Tolerances (per output, against the float64 oracle on the same dtype-rounded inputs):
  float32        O and LSE max abs error <= 1e-5; dQ, dK, dV relative Frobenius error per
                 head <= 1e-5.
  fp16 / bf16    |O - O_ref| <= 2e-2 + 2e-2 |O_ref| elementwise; LSE max abs error <= 5e-3;
                 dQ, dK, dV relative Frobenius error per head <= 3e-2.
  Every output must be finite where the oracle's is (rows with an empty allowed set: O = 0,
  LSE = -inf on both sides).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as ref
from oracle import masks
from synth import bitmap_mask, draw_head, pack_bitmap

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda", dtype=TORCH_DTYPE[dtype])


def head_inputs(wl, heads=None):
    """numpy [B,H,n,d] (rounded) for q, k, v, do, drawn head by head."""
    out = {}
    for t in ("q", "k", "v", "do"):
        arr = np.empty((wl.B, wl.H, wl.n, wl.d), np.float32)
        for bh in range(wl.heads):
            arr[bh // wl.H, bh % wl.H] = draw_head(wl, t, bh)
        out[t] = arr
    return out


def mask_for(wl, allowed=None):
    """(oracle mask function, device words or None, packed numpy words or None)."""
    if wl.mask == "bitmap":
        a = bitmap_mask(wl.n, wl.seed) if allowed is None else allowed
        words = pack_bitmap(a)
        return masks.bitmap(words, wl.n), torch.from_numpy(words.view(np.int32)).cuda(), words
    return masks.for_kind(wl.mask, wl.n), None, None


def tol_fwd(dtype):
    return (1e-5, 0.0, 1e-5) if dtype == "f32" else (2e-2, 2e-2, 5e-3)


def tol_grad(dtype):
    return 1e-5 if dtype == "f32" else 3e-2


def check_forward(o, lse, Y, L, dtype, what=""):
    """Element-wise checks of O and LSE (numpy float64 references)."""
    atol, rtol, ltol = tol_fwd(dtype)
    o = o.double().cpu().numpy() if isinstance(o, torch.Tensor) else o
    lse = lse.double().cpu().numpy() if isinstance(lse, torch.Tensor) else lse
    assert o.shape == Y.shape and lse.shape == L.shape
    empty = ~np.isfinite(L)
    assert np.all(lse[empty] == -np.inf), f"{what}: empty rows must give -inf"
    assert np.all(np.isfinite(lse[~empty])), f"{what}: non-finite LSE"
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - Y)
    bad = err > atol + rtol * np.abs(Y)
    assert not bad.any(), f"{what}: O off at {np.argwhere(bad)[:5].tolist()}, max err {err.max():.3e}"
    lerr = np.abs(lse[~empty] - L[~empty]).max(initial=0.0)
    assert lerr <= ltol, f"{what}: LSE max err {lerr:.3e} > {ltol}"
    return err.max(), lerr


def rel_frob_per_head(got, want):
    """||got - want||_F / ||want||_F per head: the relative Frobenius error the tolerance is
    stated in.  Only a head whose exact gradient is identically zero (e.g. n = 1, where every
    probability is 1 and dQ = dK = 0 exactly; the float64 oracle then returns rounding noise,
    norms below 1e-9) is measured absolutely, ||got - want||_F."""
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    g = got.reshape(-1, *got.shape[-2:])
    w = want.reshape(-1, *want.shape[-2:])
    num = np.linalg.norm((g - w).reshape(g.shape[0], -1), axis=1)
    den = np.linalg.norm(w.reshape(w.shape[0], -1), axis=1)
    return num / np.where(den < 1e-9, 1.0, den)


def check_grads(grads, refs, dtype, what=""):
    tol = tol_grad(dtype)
    worst = 0.0
    for name, got, want in zip(("dQ", "dK", "dV"), grads, refs):
        assert torch.isfinite(got).all(), f"{what}: non-finite {name}"
        e = rel_frob_per_head(got, want)
        worst = max(worst, float(e.max()))
        assert e.max() <= tol, f"{what}: {name} rel Frobenius {e.max():.3e} > {tol}"
    return worst


def oracle_forward(inp, wl, mk, heads=None):
    return ref.forward(inp["q"], inp["k"], inp["v"], wl.c, mk, heads)


def oracle_backward(inp, wl, mk, heads=None):
    return ref.backward(inp["q"], inp["k"], inp["v"], wl.c, mk, inp["do"], heads)

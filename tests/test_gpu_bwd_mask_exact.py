"""Bit-exact checks of the allowed-key sets that the backward kernels apply.

The reverse procedure of "Exact tiled attention and memory-aware differentiation" recomputes
every score block with the same fixed allowed sets A_i as the forward.  The forward's mask is
fingerprinted elsewhere (c = 0, keys encoded in binary); these tests read the mask each
backward kernel applied straight out of its outputs, one element per (query, key) pair.

Head h of a call covers the window W_h = [w h, w h + w) (w = d, so one-hot rows fit) and
one input is one-hot inside the window and zero outside it:

  dV  (key-tile kernel)    dO_i = e_{i - w h} for i in W_h:  dV[h][j, a] = p_{wh+a, j}
  dK  (key-tile kernel)    Q_i  = e_{i - w h} for i in W_h:  dK[h][j, a] = c γ_{wh+a, j}
  dQ  (query-tile kernel)  K_j  = e_{j - w h} for j in W_h:  dQ[h][i, b] = c γ_{i, wh+b}

with p_ij = exp(s_ij - LSE_i) and γ_ij = p_ij (dO_i . V_j - D_i) for allowed keys and
exactly 0 for the others.  Each output element is then a single product (the other terms
are exact zeros), so rounding can neither create nor cancel it: a disallowed pair must read
exactly 0, an allowed pair nonzero.  With ceil(n / w) heads every (query, key) pair of the
n x n mask is read once by each kernel.  One key wrongly admitted or dropped for one row in
either kernel flips one element.

An allowed pair may read 0 only where its exact value (the oracle's) vanishes (a row with a
single allowed key has p = 1 and dO_i.V_j = D_i, so γ = 0) or is below what the output type
can represent after the 16-bit rounding of γ (fp16: c γ < 2^-21); such pairs are counted and
must stay rare.  The dV readout is also compared by value with the oracle's p.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea
from oracle import attention as ref
from oracle import masks
from synth import Workload, bitmap_mask, draw_head, pack_bitmap, random_allowed

from helpers import to_dev

pytestmark = pytest.mark.gpu

# exact values below this may round to zero in the output type (fp16 subnormals)
TINY = {"f32": 0.0, "bf16": 0.0, "f16": 2.0 ** -21}
P_RTOL = {"f32": 1e-5, "bf16": 1e-2, "f16": 4e-3}


def _mask(mask, n, seed=7):
    """(oracle mask function, device words or None).  The bitmap mixes skipped, partial and
    whole 128 x 128 tiles: a 96-key band, kept 64 x 64 blocks, sparse extra keys in the first
    half of the rows, and one tile with every key allowed."""
    if mask != "bitmap":
        return masks.for_kind(mask, n), None
    a = bitmap_mask(n, seed, window=96, block=64, keep=0.3)
    extra = random_allowed(n, seed, keep=0.03, diagonal=False)
    extra[n // 2:] = False
    a |= extra
    a[:128, 256:384] = True
    words = pack_bitmap(a)
    return masks.bitmap(words, n), torch.from_numpy(words.view(np.int32)).cuda()


def _draw(seed, H, n, d, dtype):
    wl = Workload("bwd_mask", seed, 1, H, n, d, dtype, "none", 1.0 / np.sqrt(d))
    return {t: np.stack([draw_head(wl, t, h) for h in range(H)])[None] for t in ("q", "k", "v", "do")}


def _one_hot_windows(H, n, w):
    """[1, H, n, w]: head h holds e_{i - w h} in rows i of W_h, zeros elsewhere."""
    x = np.zeros((1, H, n, w), np.float32)
    for h in range(H):
        rows = np.arange(w * h, min(w * h + w, n))
        x[0, h, rows, rows - w * h] = 1.0
    return x


def _run(inp, dtype, c, mask, bits, kvb):
    dev = {t: to_dev(inp[t], dtype) for t in inp}
    o, lse = ea.attn_fwd(dev["q"], dev["k"], dev["v"], c, mask=mask, mask_bits=bits,
                         kv_block=kvb)
    grads = ea.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], c, mask=mask,
                        mask_bits=bits, kv_block=kvb)
    assert ea.attn_device_status() == ea.ATTN_OK
    return [g[0].double().cpu().numpy() for g in grads]


def _oracle(inp, c, allowed, h):
    q, k, v, g = (inp[t][0, h] for t in ("q", "k", "v", "do"))
    p, gamma, _, _ = ref.probabilities_and_gamma(q, k, v, c, allowed, g)
    return p, c * gamma


def _check_pattern(got, want_val, allowed_pairs, tiny, what):
    """got, want_val, allowed_pairs: arrays of one head's readout (same shape)."""
    disallowed_nonzero = (~allowed_pairs) & (got != 0)
    assert not disallowed_nonzero.any(), \
        f"{what}: nonzero at disallowed pairs {np.argwhere(disallowed_nonzero)[:5].tolist()}"
    # exact zeros of γ (a row with one allowed key has p = 1 and dO.V_j = D_i) and values the
    # output type cannot hold may read 0
    floor = max(tiny, 1e-6 * float(np.abs(want_val).max(initial=0.0)))
    representable = allowed_pairs & (np.abs(want_val) > floor)
    missing = representable & (got == 0)
    assert not missing.any(), f"{what}: zero at allowed pairs {np.argwhere(missing)[:5].tolist()}"
    exempt = int((allowed_pairs & ~representable).sum())
    assert exempt <= max(2, allowed_pairs.sum() // 200), f"{what}: {exempt} unrepresentable pairs"


def _cases():
    out = []
    kvbs = (32, 64, 128)
    for dtype in ("bf16", "f16", "f32"):
        for mask in ("causal", "bitmap", "none"):
            for d in (128, 64):
                for t, n in enumerate((77, 300, 513)):
                    out.append((dtype, mask, d, n, kvbs[(t + (d == 64)) % 3]))
    return out


@pytest.mark.parametrize("dtype,mask,d,n,kvb", _cases())
def test_backward_masks_bit_exact(dtype, mask, d, n, kvb):
    ea.load()
    w = d
    H = -(-n // w)
    c = 1.0 / np.sqrt(d)
    mk, bits = _mask(mask, n)
    allowed = mk(0, np.arange(n))  # one mask shared by every head
    base = _draw(31 + n, H, n, d, dtype)
    hot = _one_hot_windows(H, n, w)

    # dV: upstream gradients one-hot in the window -> dV[h][j, a] = p_{wh+a, j}
    inp = dict(base, do=hot)
    _, _, dv = _run(inp, dtype, c, mask, bits, kvb)
    for h in range(H):
        rows = np.arange(w * h, min(w * h + w, n))
        p, _ = _oracle(inp, c, allowed, h)
        got = dv[h][:, : rows.size]
        want = p[rows].T
        pairs = allowed[rows].T
        _check_pattern(got, want, pairs, 0.0, f"dV head {h}")
        assert not dv[h][:, rows.size:].any()
        err = np.abs(got - want)[pairs] / want[pairs]
        assert err.max() <= P_RTOL[dtype], f"dV head {h}: p off by {err.max():.2e} (relative)"

    # dK: queries one-hot in the window -> dK[h][j, a] = c γ_{wh+a, j}
    inp = dict(base, q=hot)
    _, dk, _ = _run(inp, dtype, c, mask, bits, kvb)
    for h in range(H):
        rows = np.arange(w * h, min(w * h + w, n))
        _, cg = _oracle(inp, c, allowed, h)
        _check_pattern(dk[h][:, : rows.size], cg[rows].T, allowed[rows].T, TINY[dtype],
                       f"dK head {h}")
        assert not dk[h][:, rows.size:].any()

    # dQ: keys one-hot in the window -> dQ[h][i, b] = c γ_{i, wh+b}
    inp = dict(base, k=hot)
    dq, _, _ = _run(inp, dtype, c, mask, bits, kvb)
    for h in range(H):
        keys = np.arange(w * h, min(w * h + w, n))
        _, cg = _oracle(inp, c, allowed, h)
        _check_pattern(dq[h][:, : keys.size], cg[:, keys], allowed[:, keys], TINY[dtype],
                       f"dQ head {h}")
        assert not dq[h][:, keys.size:].any()

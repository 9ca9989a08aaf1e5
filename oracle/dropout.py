"""Dropout on the attention probabilities with a replayed realised mask, in float64 (test
infrastructure only).

The pages' base procedure has no dropout and require of any dropout extension that its
reverse pass reuse the realised mask of the forward ("Exact tiled attention and
memory-aware differentiation", the reverse procedure and the closing remark on rounding):
a different mask differentiates a different function.  The library's reading, which this
module restates:

* Mask.  For head index bh (b·H + h), query row i and key j, the generator is
  Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
  1, 2, 3", SC 2011) with counter (⌊i/4⌋, ⌊j/4⌋, bh, 0) and key (seed mod 2^32,
  ⌊seed / 2^32⌋): one call decides the 4 x 4 patch of pairs with those row and key groups.
  Word i mod 4 of its output belongs to row i, and byte j mod 4 of that word (bits
  8 (j mod 4) .. 8 (j mod 4) + 7) to key j; the pair is kept iff that byte ≥ t, the 8-bit
  threshold t = ⌊p·256 + 1/2⌋.  The drop probability is therefore p' = t / 256 (p rounded to
  a multiple of 1/256), and kept probabilities are scaled by 1/(1 − p').  Integer arithmetic
  end to end, so the mask is the same bit for bit wherever it is drawn.
* Forward.  P_ij = exp(s_ij − LSE_i) as without dropout (LSE is not changed by dropout);
  O_i = Σ_j P_ij M_ij V_j / (1 − p').
* Reverse, for upstream G: with P̃ = P∘M/(1 − p'), dV = P̃ᵀ G;  dP̃_ij = G_i·V_j;
  D_i = G_i·O_i (= Σ_j P̃_ij dP̃_ij);  dS_ij = P_ij (M_ij dP̃_ij/(1 − p') − D_i);
  dQ = c·dS K, dK = c·dSᵀ Q.  This is the chain rule through O = (P∘M/(1−p')) V and the
  softmax, the mask held fixed.
"""
from __future__ import annotations

import math

import numpy as np

# Philox4x32 constants of the publication: round multipliers and the key's Weyl increments.
_M0, _M1 = 0xD2511F53, 0xCD9E8D57
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
_MASK32 = 0xFFFFFFFF


def philox4x32(ctr, key, rounds=10):
    """Philox4x32 with ``rounds`` rounds.  ``ctr``: uint32 array [..., 4]; ``key``: two ints.
    Returns uint32 [..., 4]."""
    c = np.asarray(ctr, dtype=np.uint64) & _MASK32
    c0, c1, c2, c3 = (c[..., t].copy() for t in range(4))
    k0, k1 = int(key[0]) & _MASK32, int(key[1]) & _MASK32
    for r in range(rounds):
        if r:
            k0, k1 = (k0 + _W0) & _MASK32, (k1 + _W1) & _MASK32
        p0 = c0 * np.uint64(_M0)  # exact: both factors < 2^32
        p1 = c2 * np.uint64(_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK32)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def threshold(p):
    """8-bit drop threshold ⌊p·256 + 1/2⌋ (halves round up); p must leave some pairs kept
    (threshold at most 255)."""
    if not 0.0 <= p < 1.0:
        raise ValueError("drop probability must be in [0, 1)")
    t = int(math.floor(p * 256.0 + 0.5))
    if t > 255:
        raise ValueError("drop probability rounds to 1 at 1/256 resolution")
    return t


def effective_p(p):
    """The drop probability the mask realises: the threshold over 256."""
    return threshold(p) / 256.0


def keep_mask(seed, bh, rows, n, p):
    """Kept pairs of head ``bh`` for query ``rows`` and keys 0..n-1: bool [len(rows), n]."""
    rows = np.asarray(rows, dtype=np.int64)
    groups = (n + 3) // 4
    ctr = np.zeros((rows.size, groups, 4), dtype=np.uint64)
    ctr[..., 0] = (rows // 4)[:, None]
    ctr[..., 1] = np.arange(groups)[None, :]
    ctr[..., 2] = bh
    words = philox4x32(ctr, (seed & _MASK32, (seed >> 32) & _MASK32))  # [rows, groups, 4]
    mine = np.take_along_axis(words, (rows % 4)[:, None, None].repeat(groups, axis=1), axis=2)[..., 0]
    j = np.arange(n)
    byte = (mine[:, j // 4].astype(np.uint64) >> (8 * (j % 4)).astype(np.uint64)) & np.uint64(0xFF)
    return byte >= np.uint64(threshold(p))


def forward_rows(q, k, v, c, allowed, keep, p):
    """O, LSE of one head's query rows ``q`` under dropout with kept pairs ``keep``."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    s = np.where(allowed, float(c) * (q @ k.T), -np.inf)
    m = s.max(axis=1)
    nonempty = np.isfinite(m)
    e = np.exp(s - np.where(nonempty, m, 0.0)[:, None])
    ell = e.sum(axis=1)
    safe = np.where(nonempty, ell, 1.0)
    P = e / safe[:, None]
    y = ((P * keep) @ v) / (1.0 - effective_p(p))
    y[~nonempty] = 0.0
    lse = np.where(nonempty, m + np.log(safe), -np.inf)
    return y, lse


def probabilities_and_gamma(q, k, v, c, allowed, keep, p, G):
    """P [n,n] (undropped probabilities), dP̃ = G Vᵀ [n,n] and γ = dS [n,n] of one head under
    dropout with kept pairs ``keep``: γ_ij = P_ij (M_ij dP̃_ij/(1 − p') − D_i)."""
    q, k, v, G = (np.asarray(x, dtype=np.float64) for x in (q, k, v, G))
    y, lse = forward_rows(q, k, v, c, allowed, keep, p)
    s = np.where(allowed, float(c) * (q @ k.T), -np.inf)
    fin = np.isfinite(lse)
    P = np.where(fin[:, None], np.exp(s - np.where(fin, lse, 0.0)[:, None]), 0.0)
    dPt = G @ v.T
    D = (G * y).sum(axis=1)
    gamma = P * (keep * dPt / (1.0 - effective_p(p)) - D[:, None])
    return P, dPt, gamma


def backward_head(q, k, v, c, allowed, keep, p, G):
    """dQ, dK, dV of one head under dropout (the mask ``keep`` replayed)."""
    q, k, v, G = (np.asarray(x, dtype=np.float64) for x in (q, k, v, G))
    y, lse = forward_rows(q, k, v, c, allowed, keep, p)
    s = np.where(allowed, float(c) * (q @ k.T), -np.inf)
    fin = np.isfinite(lse)
    P = np.where(fin[:, None], np.exp(s - np.where(fin, lse, 0.0)[:, None]), 0.0)
    pe = effective_p(p)
    Pt = P * keep / (1.0 - pe)
    dV = Pt.T @ G
    dPt = G @ v.T
    D = (G * y).sum(axis=1)
    dS = P * (keep * dPt / (1.0 - pe) - D[:, None])
    dQ = float(c) * dS @ k
    dK = float(c) * dS.T @ q
    return dQ, dK, dV

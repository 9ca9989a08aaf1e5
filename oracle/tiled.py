"""The block-by-block algorithm of "Exact tiled attention and memory-aware differentiation"
in float64 (test infrastructure only).

Definitions followed (that page, "Stable summary of an attention key block"):
  the summary of a nonempty key set S for query row i is Σ_i(S) = (m, ℓ, z) with
  m = max_{j∈S} s_ij, ℓ = Σ_{j∈S} e^{s_ij - m}, z = Σ_{j∈S} e^{s_ij - m} v_j;
  the empty set has the separate state ⊥ (here ``BOTTOM``);
  two summaries of disjoint sets merge as m' = max(m_S, m_T),
  ℓ' = e^{m_S-m'} ℓ_S + e^{m_T-m'} ℓ_T, z' = e^{m_S-m'} z_S + e^{m_T-m'} z_T.

Algorithm followed (same page, "Exact tiled softmax attention with block-recomputed
vector-Jacobian products"):
  forward — key blocks J_t = {(t-1)b+1, .., min(tb, n)} in order; per row start from ⊥; skip
  a block whose allowed part I = J_t ∩ A_i is empty; otherwise take Σ_i(I) and copy it
  into an empty state or merge it into the current one; at the end Y_i = z_i / ℓ_i and
  (m_i, ℓ_i) are retained.
  reverse — zero dQ, dK, dV; per row δ_i = G_i·Y_i; per block and allowed key recompute
  s_ij, p_ij = e^{s_ij - m_i}/ℓ_i, γ_ij = p_ij (G_i·V_j - δ_i), then add c γ_ij K_j to dQ_i,
  c γ_ij Q_i to dK_j and p_ij G_i to dV_j.

Key-sharded forward (same page, the merge read as combining shards): the summaries of
disjoint key sets merge into the summary of their union, so a row's keys can be cut into
shares, each share summarised on its own, and the shares merged.  ``merge_normalised`` takes
the shares in the normalised form a kernel writes (O_g = z_g / ℓ_g, LSE_g = m_g + ln ℓ_g).

Indices here are 0-based.  The streaming-softmax recurrence of "The Arithmetic of
Intelligence", chapter 12 (running max m, running sum ℓ, rescale by e^{m-m'}) is the same
merge with a block's own summary, so ``streaming_normaliser`` reuses ``merge``.
"""
from __future__ import annotations

import math

import numpy as np

BOTTOM = None  # summary of the empty key set


def block_summary(s, vrows):
    """Σ(S) = (m, ℓ, z) for the scores ``s`` of a nonempty key set and its value rows."""
    s = np.asarray(s, dtype=np.float64).reshape(-1)
    if s.size == 0:
        return BOTTOM
    m = float(s.max())
    w = np.exp(s - m)
    z = w @ np.asarray(vrows, dtype=np.float64).reshape(s.size, -1)
    return (m, float(w.sum()), z)


def merge(a, b):
    """Σ(S) ⋆ Σ(T) for disjoint S, T; ⊥ acts as the identity."""
    if a is BOTTOM:
        return b
    if b is BOTTOM:
        return a
    ma, la, za = a
    mb, lb, zb = b
    m = max(ma, mb)
    ea = math.exp(ma - m)
    eb = math.exp(mb - m)
    return (m, ea * la + eb * lb, ea * za + eb * zb)


def streaming_normaliser(blocks):
    """Running (m, ℓ) after scores arrive block by block (values taken as zero-width)."""
    state = BOTTOM
    for blk in blocks:
        blk = np.asarray(blk, dtype=np.float64)
        state = merge(state, block_summary(blk, np.zeros((blk.size, 0))))
    return state[0], state[1]


def key_blocks(n, b):
    """J_t, t = 1..ceil(n/b), as 0-based index ranges."""
    return [np.arange(t * b, min((t + 1) * b, n)) for t in range((n + b - 1) // b)]


def forward_head(q, k, v, c, allowed, b):
    """Y, m, ℓ of one head by the tiled forward procedure.  ``allowed`` is bool [n, n]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n = q.shape[0]
    Y = np.zeros((n, v.shape[1]))
    m = np.full(n, -np.inf)
    ell = np.zeros(n)
    blocks = key_blocks(k.shape[0], b)
    for i in range(n):
        state = BOTTOM
        for J in blocks:
            I = J[allowed[i, J]]
            if I.size == 0:
                continue
            s = float(c) * (k[I] @ q[i])
            state = merge(state, block_summary(s, v[I]))
        if state is BOTTOM:  # empty A_i: outside the pages' domain; library reading
            continue
        m[i], ell[i], z = state
        Y[i] = z / ell[i]
    return Y, m, ell


def reverse_head(q, k, v, c, allowed, b, Y, m, ell, G):
    """dQ, dK, dV of one head by the per-element reverse procedure."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    n = q.shape[0]
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    blocks = key_blocks(k.shape[0], b)
    for i in range(n):
        if not np.isfinite(m[i]):
            continue
        delta = float(G[i] @ Y[i])
        for J in blocks:
            for j in J[allowed[i, J]]:
                s = float(c) * float(q[i] @ k[j])
                p = math.exp(s - m[i]) / ell[i]
                gamma = p * (float(G[i] @ v[j]) - delta)
                dQ[i] += c * gamma * k[j]
                dK[j] += c * gamma * q[i]
                dV[j] += p * G[i]
    return dQ, dK, dV


def merge_normalised(parts):
    """(O, LSE) of the union of disjoint key sets from the sets' normalised results.

    ``parts`` holds (O_g, LSE_g) for one query row: O_g = z_g / ℓ_g and LSE_g = m_g + ln ℓ_g
    of key set S_g, or LSE_g = -inf for a set with no allowed key (then O_g is ignored).  The
    summaries (m, ℓ, z) and (m + ln ℓ, 1, z / ℓ) give the same z / ℓ and the same m + ln ℓ, the
    two things the forward keeps, so a part enters ``merge`` as (LSE_g, 1, O_g) and an empty
    part as ⊥.  Returns O = z / ℓ and LSE = m + ln ℓ of the merged summary, or (zeros, -inf)
    when every part is empty.
    """
    state = BOTTOM
    width = None
    for o_g, lse_g in parts:
        o_g = np.asarray(o_g, dtype=np.float64).reshape(-1)
        width = o_g.size
        if lse_g == -math.inf:
            continue
        state = merge(state, (float(lse_g), 1.0, o_g))
    if state is BOTTOM:
        return np.zeros(width or 0), -math.inf
    m, ell, z = state
    return z / ell, m + math.log(ell)


def key_shares(reach, parts, b):
    """Key-index ranges of ``parts`` contiguous shares of the first ``reach`` key blocks of
    size b (equal block counts, the last shares possibly short or empty)."""
    share = -(-reach // parts)
    out = []
    for g in range(parts):
        lo, hi = min(g * share, reach), min((g + 1) * share, reach)
        out.append(np.arange(lo * b, hi * b))
    return out

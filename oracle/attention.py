"""Dense masked softmax attention and its gradient in float64 (test infrastructure only).

The definition, as stated in "Exact tiled attention and memory-aware differentiation"
(definition of the stable summary; exactness theorem) and in the scaled dot-product
attention section of "Bellek Duvarının Fiziği" (S = QKᵀ/√d_k, P = softmax(S), O = PV):

    s_ij  = c · Σ_r Q_ir K_jr                       for j in A_i (excluded keys: -inf)
    m_i   = max_{j∈A_i} s_ij
    ℓ_i   = Σ_{j∈A_i} exp(s_ij - m_i)
    Y_i   = Σ_{j∈A_i} exp(s_ij - m_i) V_j / ℓ_i
    LSE_i = m_i + ln ℓ_i   (natural log; the retained row statistic in one number)

The reverse map for an upstream G (exactness theorem, proof steps 4-5):

    δ_i   = Σ_a G_ia Y_ia
    p_ij  = exp(s_ij - LSE_i)
    γ_ij  = p_ij (Σ_a G_ia V_ja - δ_i)
    dQ    = c · γ K,   dK = c · γᵀ Q,   dV = pᵀ G

Every array is materialised (the whole n x n score matrix of one head); matrix products
go through numpy's BLAS in float64.  A row whose allowed set is empty has no defined
output (the pages assert no convention); the library's reading is Y_i = 0, LSE_i = -inf
and no gradient contribution, and the oracle follows it.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def masked_scores(q, k, c, allowed):
    """s = c·q kᵀ on allowed entries, -inf elsewhere.  q [r,d], k [n,d], allowed [r,n]."""
    s = float(c) * (_f64(q) @ _f64(k).T)
    return np.where(allowed, s, -np.inf)


def forward_rows(q, k, v, c, allowed):
    """Y, LSE, m, ℓ for the query rows ``q`` of one head."""
    s = masked_scores(q, k, c, allowed)
    m = s.max(axis=1)
    nonempty = np.isfinite(m)
    shift = np.where(nonempty, m, 0.0)
    e = np.exp(s - shift[:, None])  # exp(-inf) = 0 for excluded keys
    ell = e.sum(axis=1)
    safe = np.where(nonempty, ell, 1.0)
    y = (e @ _f64(v)) / safe[:, None]
    y[~nonempty] = 0.0
    lse = np.where(nonempty, m + np.log(safe), -np.inf)
    return y, lse, m, ell


def forward(Q, K, V, c, mask, heads=None):
    """Y [B,H,n,v] and LSE [B,H,n] over all (or the listed flat) heads."""
    B, H, n, _ = Q.shape
    Y = np.zeros(Q.shape[:3] + (V.shape[-1],), dtype=np.float64)
    L = np.full(Q.shape[:3], -np.inf)
    rows = np.arange(n)
    for bh in (range(B * H) if heads is None else heads):
        b, h = divmod(bh, H)
        y, lse, _, _ = forward_rows(Q[b, h], K[b, h], V[b, h], c, mask(bh, rows))
        Y[b, h], L[b, h] = y, lse
    return Y, L


def probabilities_and_gamma(q, k, v, c, allowed, g):
    """p [n,n] and γ [n,n] of one head (the reverse map's per-element quantities), plus the
    forward's Y and LSE.  Both are exactly 0 where the key is not allowed."""
    y, lse, _, _ = forward_rows(q, k, v, c, allowed)
    s = masked_scores(q, k, c, allowed)
    finite = np.isfinite(lse)
    p = np.exp(s - np.where(finite, lse, 0.0)[:, None])
    p[~finite] = 0.0
    g = _f64(g)
    delta = (g * y).sum(axis=1)
    dp = g @ _f64(v).T
    gamma = p * (dp - delta[:, None])
    return p, gamma, y, lse


def backward_head(q, k, v, c, allowed, g):
    """dQ, dK, dV of Φ = Σ G∘Y for one head, plus the forward's Y and LSE."""
    p, gamma, y, lse = probabilities_and_gamma(q, k, v, c, allowed, g)
    g = _f64(g)
    dq = float(c) * (gamma @ _f64(k))
    dk = float(c) * (gamma.T @ _f64(q))
    dv = p.T @ g
    return dq, dk, dv, y, lse


def backward(Q, K, V, c, mask, G, heads=None):
    """dQ, dK, dV [B,H,n,d] over all (or the listed flat) heads."""
    B, H, n, _ = Q.shape
    dQ = np.zeros(Q.shape, dtype=np.float64)
    dK = np.zeros(K.shape, dtype=np.float64)
    dV = np.zeros(V.shape, dtype=np.float64)
    rows = np.arange(n)
    for bh in (range(B * H) if heads is None else heads):
        b, h = divmod(bh, H)
        dq, dk, dv, _, _ = backward_head(Q[b, h], K[b, h], V[b, h], c, mask(bh, rows), G[b, h])
        dQ[b, h], dK[b, h], dV[b, h] = dq, dk, dv
    return dQ, dK, dV

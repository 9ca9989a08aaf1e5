"""FP8 (E4M3) rounding and the FP8 forward's reference with its error bound, in float64 (test
infrastructure only).

E4M3 (the 8-bit format with 1 sign, 4 exponent and 3 fraction bits, exponent bias 7, no
infinities): normal values 2^e (1 + f/8) for e in [-6, 8] (the largest, 448, is 1.75 · 2^8),
subnormal values f · 2^-9 for f in 1..7.  ``round_e4m3`` rounds to the nearest such value,
ties to the even fraction, and saturates finite overflow at ±448 (the conversion the FP8
forward applies to its probabilities).

The FP8 forward computes exact tiled attention on the dequantized inputs Q = sq q8, K = sk
k8, V = sv v8, except that each probability enters the P·V product rounded to E4M3 after
scaling by 2^8 relative to the running maximum.  Rounding P' = 2^8 e^{s - m} changes it by at
most max(2^-4 P', 2^-10) (half an ulp in the normal range, half the subnormal step below), so
the output moves by at most
    bound_ia = Σ_j (2^-4 P_ij + 2^-18) |V_ja|          (P the exact normalised probabilities)
since the normaliser Σ_j P'_j is at least 2^8 (the row maximum contributes 2^8).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def round_e4m3(x):
    """Nearest E4M3 value (ties to even fraction), finite overflow saturated to ±448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)  # below 2^-6 the spacing stays 2^-9 (subnormals)
    ulp = np.exp2(e - 3.0)
    q = np.round(a / ulp) * ulp  # numpy rounds halves to even
    q = np.minimum(q, E4M3_MAX)
    return np.where(a > 0, np.sign(x) * q, 0.0 * x)


def quantize(x, scale):
    """Values x / scale rounded to E4M3, and their dequantized values (E4M3 value · scale)."""
    q = round_e4m3(np.asarray(x, dtype=np.float64) / scale)
    return q, q * scale


def forward_rows_bound(q, k, v, c, allowed):
    """Exact Y, LSE of one head (dequantized inputs) and the elementwise FP8 rounding bound."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    s = np.where(allowed, float(c) * (q @ k.T), -np.inf)
    m = s.max(axis=1)
    fin = np.isfinite(m)
    e = np.exp(s - np.where(fin, m, 0.0)[:, None])
    ell = e.sum(axis=1)
    P = e / np.where(fin, ell, 1.0)[:, None]
    P[~fin] = 0.0
    Y = P @ v
    lse = np.where(fin, m + np.log(np.where(fin, ell, 1.0)), -np.inf)
    bound = (2.0 ** -4 * P + 2.0 ** -18 * allowed) @ np.abs(v)
    return Y, lse, bound

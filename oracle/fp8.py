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

Block scaling and incoherent processing (the FP8 variant "Bellek Duvarının Fiziği" names for
FlashAttention-3: scales per block, random sign multipliers).  Readings taken here:

* A block is ``rows`` = 128 consecutive rows of one head's Q, K or V (the last one ragged),
  with one float32 scale: absmax / 448, or 1 for an all-zero block.  The codes are taken in
  float32, the precision of the GPU path: inv = fl32(448 / absmax), code = E4M3(fl32(x · inv)).
* Incoherent processing multiplies the columns of Q and K by random signs σ (an input) and
  applies the Walsh–Hadamard matrix H_d (Sylvester's construction, d a power of two):
  Q' = (Q ∘ σ) H_d, K' = (K ∘ σ) H_d.  H_d H_dᵀ = d I, so Q' K'ᵀ = d Q Kᵀ; the factor 1/d is
  folded into Q's scales.  V is not rotated.
* Within the P·V product a key block's value scale sv_J enters through the probabilities:
  the kernel rounds P'_ij = 2^8 e^{s_ij - m_i} r_J to E4M3, r_J = sv_J / max_J sv_J <= 1, and
  multiplies z by max_J sv_J at the end.  The same argument as above gives
      bound_ia = Σ_j (2^-4 P_ij + 2^-18 / r_J(j)) |V_ja|.
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


def forward_rows_bound(q, k, v, c, allowed, ratio=None):
    """Exact Y, LSE of one head (dequantized inputs) and the elementwise FP8 rounding bound.

    ``ratio`` (one entry per key, default all ones) is r_J of the key's value block: the
    probabilities of that block are rounded as 2^8 e^{s - m} r_J (block-scaled values)."""
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
    r = np.ones(k.shape[0]) if ratio is None else np.asarray(ratio, dtype=np.float64)
    bound = (2.0 ** -4 * P + 2.0 ** -18 * allowed / r[None, :]) @ np.abs(v)
    return Y, lse, bound


def hadamard(d):
    """Sylvester's Walsh–Hadamard matrix of order d (a power of two): H_1 = [1],
    H_2m = [[H_m, H_m], [H_m, -H_m]]."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate(x, signs):
    """Incoherent processing of the rows of x [.., d]: (x ∘ σ) H_d, in float64."""
    x = np.asarray(x, dtype=np.float64)
    return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(x.shape[-1])


def quantize_blocks(x, rows=128, divide=1.0):
    """Block quantization of one head's rows x [n, d] (float32-representable values).

    Returns (codes [n, d] as E4M3 values, scales [ceil(n / rows)] as float32 values):
    per block absmax; scale = fl32(absmax / 448) / divide (1 for a zero block); codes =
    E4M3(fl32(x · fl32(448 / absmax))).  ``divide`` is a power of two folded into the scale
    (d for incoherently processed queries)."""
    x32 = np.asarray(x, dtype=np.float32)
    n = x32.shape[0]
    nb = (n + rows - 1) // rows
    codes = np.zeros(x32.shape, dtype=np.float64)
    scales = np.zeros(nb, dtype=np.float64)
    for b in range(nb):
        blk = x32[b * rows:(b + 1) * rows]
        amax = np.float32(np.max(np.abs(blk))) if blk.size else np.float32(0)
        if amax == 0:
            scales[b] = 1.0 / divide
            continue
        inv = np.float32(448.0) / amax
        scales[b] = float(amax / np.float32(448.0)) / divide
        codes[b * rows:(b + 1) * rows] = round_e4m3((blk * inv).astype(np.float64))
    return codes, scales


def block_quantized_head(q, k, v, signs=None, rows=128):
    """The block-scaled FP8 operands of one head and the exact inputs they stand for.

    Q and K are incoherently processed when ``signs`` is given (rounded to float32 after the
    float64 rotation).  Returns a dict with the codes (q8, k8, v8), the per-block scales (sq,
    sk, sv), the dequantized operands (Q~ = sq q8, K~ = sk k8, V~ = sv v8, with Q~ K~ᵀ
    approximating Q Kᵀ) and r, the per-key ratio sv_J / max sv."""
    d = q.shape[-1]
    if signs is not None:
        qx = rotate(q, signs).astype(np.float32)
        kx = rotate(k, signs).astype(np.float32)
        div = float(d)
    else:
        qx, kx, div = np.asarray(q, np.float32), np.asarray(k, np.float32), 1.0
    q8, sq = quantize_blocks(qx, rows, div)
    k8, sk = quantize_blocks(kx, rows)
    v8, sv = quantize_blocks(np.asarray(v, np.float32), rows)
    per_row = lambda s, n: np.repeat(s, rows)[:n]
    n_q, n_k = q.shape[0], k.shape[0]
    return {"q8": q8, "k8": k8, "v8": v8, "sq": sq, "sk": sk, "sv": sv,
            "q": q8 * per_row(sq, n_q)[:, None], "k": k8 * per_row(sk, n_k)[:, None],
            "v": v8 * per_row(sv, n_k)[:, None], "r": per_row(sv / sv.max(), n_k)}

"""Seeded synthetic workloads for exact tiled attention.

Every tensor is drawn per (tensor, head) from its own PCG64 stream keyed by
``SeedSequence([workload seed, tensor index, flat head index])``, so any single head can
be regenerated without drawing the rest.  Entries are iid N(0,1) in float32, optionally
scaled (the query scale of the fp16 overflow workload), then rounded to the run's dtype by
round-to-nearest-even and returned as float32 values that the dtype represents exactly.

The allowed-key bitmap of the block-sparse workload is a union of a 256-key sliding window,
64x64 key blocks kept iid with probability 0.3, and the diagonal, shared by all heads.  The
packed form is the library's caller-owned mask storage: row-major ``[n][row_words]`` uint32,
key ``j`` allowed iff bit ``j % 32`` of word ``j // 32`` is set (least significant bit first).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

TENSOR_INDEX = {"q": 0, "k": 1, "v": 2, "do": 3}


@dataclass(frozen=True)
class Workload:
    """Shape, precision, mask and scale of one synthetic attention problem."""

    name: str
    seed: int
    B: int
    H: int
    n: int
    d: int
    dtype: str  # "f32" | "f16" | "bf16"
    mask: str  # "none" | "causal" | "bitmap"
    c: float
    kv_block: int = 0  # 0: the library picks the key block
    q_scale: float = 1.0
    passes: tuple = ("fwd", "bwd")
    kv_blocks: tuple = field(default=())  # extra key-block sizes the workload must agree over

    @property
    def heads(self) -> int:
        return self.B * self.H

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _configs() -> dict:
    r = math.sqrt
    cf = {}
    cf["small_causal_f32"] = Workload("small_causal_f32", 1, 1, 1, 256, 64, "f32", "causal",
                                      1.0 / 8.0, kv_block=64)
    for d in (16, 64):
        # Q scaled by 2.5 as the workload states.  "hot" also scales c by 2.5, which puts
        # the per-row maximum score near 20-25, the range the overflow workload names.
        cf[f"overflow_f16_d{d}"] = Workload(f"overflow_f16_d{d}", 2, 1, 4, 4096, d, "f16",
                                            "causal", 1.0 / r(d), q_scale=2.5,
                                            passes=("fwd",))
        cf[f"overflow_f16_d{d}_hot"] = Workload(f"overflow_f16_d{d}_hot", 2, 1, 4, 4096, d,
                                                "f16", "causal", 2.5 / r(d), q_scale=2.5,
                                                passes=("fwd",))
    cf["train_bf16_d128"] = Workload("train_bf16_d128", 3, 8, 16, 4096, 128, "bf16", "none",
                                     1.0 / r(128))
    for n in (16384, 65536):
        cf[f"longctx_bf16_n{n}"] = Workload(f"longctx_bf16_n{n}", 4, 1, 32, n, 128, "bf16",
                                            "causal", 1.0 / r(128), passes=("fwd",))
    for dt in ("f32", "bf16"):
        cf[f"bitmap_{dt}"] = Workload(f"bitmap_{dt}", 5, 2, 8, 2048, 64, dt, "bitmap",
                                      1.0 / 8.0, kv_block=64, kv_blocks=(32, 64, 128))
    return cf


CONFIGS = _configs()


def workload(name: str) -> Workload:
    return CONFIGS[name]


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to ``dtype`` (nearest-even) and return them as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
        return u.astype(np.uint32).view(np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def draw_head(wl: Workload, tensor: str, bh: int, n: int | None = None) -> np.ndarray:
    """One head's ``[n, d]`` slice of tensor ``tensor`` ("q", "k", "v" or "do")."""
    n = wl.n if n is None else n
    ss = np.random.SeedSequence([wl.seed, TENSOR_INDEX[tensor], bh])
    g = np.random.Generator(np.random.PCG64(ss))
    x = g.standard_normal((n, wl.d), dtype=np.float32)
    if tensor == "q" and wl.q_scale != 1.0:
        x *= np.float32(wl.q_scale)
    return round_to_dtype(x, wl.dtype)


def draw_tensor(wl: Workload, tensor: str) -> np.ndarray:
    """The whole ``[B, H, n, d]`` tensor, head by head."""
    out = np.empty((wl.B, wl.H, wl.n, wl.d), dtype=np.float32)
    for bh in range(wl.heads):
        out[bh // wl.H, bh % wl.H] = draw_head(wl, tensor, bh)
    return out


def bitmap_mask(n: int, seed: int, window: int = 256, block: int = 64,
                keep: float = 0.3) -> np.ndarray:
    """Boolean ``[n, n]`` allowed-key sets: sliding window | kept blocks | diagonal."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    half = window // 2
    allowed = (j >= i - half) & (j <= i + half - 1)
    nb = -(-n // block)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 17])))
    kept = g.random((nb, nb)) < keep
    allowed |= kept[i // block, j // block]
    allowed |= i == j
    return allowed


def random_allowed(n: int, seed: int, keep: float = 0.3, diagonal: bool = True) -> np.ndarray:
    """Boolean ``[n, n]`` allowed sets with iid membership (probability ``keep``)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 29])))
    a = g.random((n, n)) < keep
    if diagonal:
        a[np.arange(n), np.arange(n)] = True
    return a


def pack_bitmap(allowed: np.ndarray, row_words: int | None = None) -> np.ndarray:
    """Pack a boolean ``[rows, n]`` mask into ``[rows, row_words]`` uint32, LSB first."""
    allowed = np.asarray(allowed, dtype=bool)
    rows, n = allowed.shape
    need = -(-n // 32)
    row_words = need if row_words is None else row_words
    if row_words < need:
        raise ValueError("row_words too small")
    padded = np.zeros((rows, row_words * 32), dtype=bool)
    padded[:, :n] = allowed
    by = np.packbits(padded, axis=1, bitorder="little")  # [rows, row_words*4] uint8
    return np.ascontiguousarray(by).view("<u4").astype(np.uint32).reshape(rows, row_words)

"""Allowed-key sets A_i for the oracle (test infrastructure only).

Each mask is a function ``allowed(bh, rows) -> bool[len(rows), n]`` giving, for head ``bh``
and query rows ``rows``, which keys are members of A_i.

* none   — every key is allowed.
* causal — key j is allowed for query i iff j <= i (0-indexed, diagonal included): the
           "Night School: fused attention" page has each word score itself and every earlier
           word (section "The table of scores").
* causal_rect — m query rows against n keys with the queries at the end of the sequence (the
           decoding reading of a key/value cache: query i stands at position i + n - m), key j
           allowed iff j <= i + n - m; m = n is the causal mask above.
* bitmap — the caller-owned packed representation of the allowed sets named in "Exact tiled
           attention and memory-aware differentiation" (algorithm inputs: membership is read
           on demand from input storage).  Row-major ``[n][row_words]`` uint32 words; key j
           is allowed iff bit (j mod 32) of word floor(j / 32) is set.  An optional per-head
           stride (in words) selects a different bitmap per flat head index.
"""
from __future__ import annotations

import numpy as np


def none(n: int):
    def allowed(bh, rows):
        rows = np.asarray(rows)
        return np.ones((rows.size, n), dtype=bool)
    return allowed


def causal(n: int):
    keys = np.arange(n)

    def allowed(bh, rows):
        rows = np.asarray(rows).reshape(-1, 1)
        return keys[None, :] <= rows
    return allowed


def causal_rect(m: int, n: int):
    keys = np.arange(n)
    off = n - m

    def allowed(bh, rows):
        rows = np.asarray(rows).reshape(-1, 1)
        return keys[None, :] <= rows + off
    return allowed


def unpack_row(words: np.ndarray, n: int) -> np.ndarray:
    """Membership of keys 0..n-1 from one row of packed words, bit by bit."""
    words = np.asarray(words, dtype=np.uint64)
    j = np.arange(n)
    return ((words[j // 32] >> (j % 32).astype(np.uint64)) & np.uint64(1)).astype(bool)


def bitmap(words: np.ndarray, n: int, head_stride_words: int = 0):
    """Mask read from packed words.  ``words`` is 1-D (flat storage) or ``[.., row_words]``."""
    flat = np.ascontiguousarray(words, dtype=np.uint32).reshape(-1)
    row_words = None if np.ndim(words) == 1 else np.shape(words)[-1]
    if row_words is None:
        raise ValueError("pass words shaped [rows, row_words]")

    j = np.arange(n)
    word_of_key = j // 32
    bit_of_key = (j % 32).astype(np.uint64)

    def allowed(bh, rows):
        rows = np.asarray(rows, dtype=np.int64).reshape(-1)
        starts = bh * head_stride_words + rows * row_words
        w = flat[starts[:, None] + word_of_key[None, :]].astype(np.uint64)
        return ((w >> bit_of_key[None, :]) & np.uint64(1)).astype(bool)
    return allowed


def dense(allowed_matrix: np.ndarray):
    """Mask given as an explicit boolean ``[n, n]`` matrix shared by all heads."""
    a = np.asarray(allowed_matrix, dtype=bool)

    def allowed(bh, rows):
        return a[np.asarray(rows).reshape(-1)]
    return allowed


def for_kind(kind: str, n: int, bits: np.ndarray | None = None, head_stride_words: int = 0):
    if kind == "none":
        return none(n)
    if kind == "causal":
        return causal(n)
    if kind == "bitmap":
        return bitmap(bits, n, head_stride_words)
    raise ValueError(kind)

"""Global-memory byte counter for one attention head (test infrastructure only).

Restates the lab of "Night School: fused attention" (section "The lab: the cannery" and
"One trip"): an emulator that counts every byte two float32 kernels request from global
memory for one head of n tokens and d numbers per head.

* fused ("crew and bench"): a crew loads a tile of query rows onto an on-chip bench, walks
  every key row and value row past it, keeps the running maximum and total on chip, and
  writes only the finished output rows (no row statistics).  The bench is small, so K and V
  are fetched again for every query tile.
* unfused (three passes): write the scores, read them back and write the shares, read the
  shares back to mix; the score and share tables each cross the memory boundary twice.  The
  score pass and the mixing pass use the same query-row tiling as the fused kernel, so they
  also fetch K (resp. V) once per tile.

The page gives the totals but not the tile height.  Reading used here: the bench holds 2048
float32 query values, so a tile has 2048 // d rows.  With that one reading the counter
reproduces all four totals the page prints for n = 4096 (d = 16: 285,736,960 vs 17,301,504;
d = 64: 538,968,064 vs 270,532,608).  No causal tile skipping is modelled, because the
printed totals imply none.
"""
from __future__ import annotations

FLOAT = 4  # bytes per float32


def tile_rows(d: int, bench_floats: int = 2048) -> int:
    return max(1, bench_floats // d)


def fused_bytes(n: int, d: int, bench_floats: int = 2048) -> int:
    rows = tile_rows(d, bench_floats)
    total = 0
    for r0 in range(0, n, rows):
        r = min(rows, n - r0)
        total += r * d * FLOAT  # load the query tile onto the bench
        total += n * d * FLOAT  # walk every key row past it
        total += n * d * FLOAT  # and every value row
        total += r * d * FLOAT  # write the finished output rows
    return total


def unfused_bytes(n: int, d: int, bench_floats: int = 2048) -> int:
    rows = tile_rows(d, bench_floats)
    total = 0
    for r0 in range(0, n, rows):  # pass 1: scores
        r = min(rows, n - r0)
        total += r * d * FLOAT + n * d * FLOAT  # query tile, all keys
        total += r * n * FLOAT  # write score rows
    total += n * n * FLOAT + n * n * FLOAT  # pass 2: read scores, write shares
    for r0 in range(0, n, rows):  # pass 3: mix
        r = min(rows, n - r0)
        total += r * n * FLOAT + n * d * FLOAT  # share rows, all values
        total += r * d * FLOAT  # write output rows
    return total

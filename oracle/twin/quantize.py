"""LUT-6 quantiser: the numpy twin of the C++ oracle (float64 with exact integer sums).

Source: "Clef-Flash-ANE-LUT6" model card, section "LUT-6 text weights": a 64-entry table per 16
output channels, fitted by k-means in one dimension for 40 iterations, whose initial centroids are
32 quantiles of the channels' weights and 32 points at equal steps from their smallest to their
largest weight.

Readings where the card is silent (each is a plain choice the rest of the card allows):
  * quantiles: the 32 probabilities (i + 1/2) / 32, i = 0..31, each taken between the two
    neighbouring order statistics by linear interpolation, x[lo] + f (x[lo+1] - x[lo]) with
    h = p (n - 1), lo = floor(h), f = h - lo.  For fp16 weights every step is exact in float64;
  * evenly spread: min + i * step, step = (max - min) / 31, i = 0..30, rounded after the
    division, the product and the sum; the 32nd value is max itself;
  * the 64 initial centroids (quantiles first, then the equal-step points) are sorted ascending by a
    stable sort, so equal values (-0 and +0 among them) keep that order.  After every round the
    centroids are sorted again the same way: equal seeds share their members with the first of
    them, which moves while the others stay, so order is not kept by itself.  Sorting changes
    only the labels (the set of centroids, and so every later round, is the same);
  * a round assigns each weight to its nearest centroid.  With ascending centroids that is the
    cell between the midpoints of neighbouring centroids, each midpoint fl(c_j + c_j+1) / 2;
    a weight exactly on a midpoint goes to the lower index, and a weight whose nearest value is
    held by several equal centroids goes to the first of them.  Each centroid with members
    moves to their mean; one without members stays;
  * the mean has a single rounding: fp16 weights are integer multiples of 2^-24, so their sum
    is an exact integer S (in units of 2^-24); the centroid is fl(fl(S) / count) * 2^-24;
  * after 40 rounds the table is the centroids rounded to fp16 (nearest, ties to even) and each
    weight's index is its nearest table entry, a tie (a midpoint, or equal entries) going to the
    lower index (the midpoints of fp16 neighbours are exact in float64);
  * weights must be finite.
"""
from __future__ import annotations

import numpy as np

from .lut6 import GROUP_ROWS, TABLE_SIZE, pack

ROUNDS = 40
FIX = 2.0 ** 24          # fp16 values are integer multiples of 2^-24
HALF = TABLE_SIZE // 2   # quantile seeds, and evenly spread seeds


def quantiles(values: np.ndarray) -> np.ndarray:
    """The 32 quantile seeds of one group, float64 ascending."""
    x = np.sort(np.asarray(values, dtype=np.float64).ravel())
    n = x.size
    out = np.empty(HALF)
    for i in range(HALF):
        h = (i + 0.5) / HALF * (n - 1)
        lo = int(np.floor(h))
        hi = min(lo + 1, n - 1)
        f = h - lo
        out[i] = x[lo] + f * (x[hi] - x[lo])
    return out


def spread(values: np.ndarray) -> np.ndarray:
    """The 32 evenly spread seeds from min to max, float64."""
    v = np.asarray(values, dtype=np.float64).ravel()
    lo, hi = float(v.min()), float(v.max())
    step = (hi - lo) / (HALF - 1)
    out = np.array([i * step + lo for i in range(HALF)])
    out[-1] = hi
    return out


def initial_table(values: np.ndarray) -> np.ndarray:
    """64 starting centroids of one group (float64, ascending)."""
    return np.sort(np.concatenate([quantiles(values), spread(values)]), kind="stable")


def assign(values: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """Nearest of ascending centroids: the cell is the number of midpoints strictly below the
    value; a cell whose centroid repeats earlier ones maps to the first of the repeats."""
    c = np.asarray(centroids, dtype=np.float64)
    mid = (c[:-1] + c[1:]) / 2.0
    cell = np.searchsorted(mid, np.asarray(values, dtype=np.float64).ravel(), side="left")
    first = np.searchsorted(c, c, side="left")
    return first[cell]


def kmeans_round(values: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """One round: assign, move each centroid with members to their mean, sort (stable)."""
    v = np.asarray(values, dtype=np.float64).ravel()
    c = np.array(centroids, dtype=np.float64)
    a = assign(v, c)
    fixed = np.rint(v * FIX).astype(np.int64)               # exact for fp16 weights
    for j in range(c.size):
        members = a == j
        count = int(members.sum())
        if count:
            total = int(fixed[members].sum())               # exact integer sum
            c[j] = (float(total) / float(count)) / FIX
    return np.sort(c, kind="stable")


def quantize_group(values: np.ndarray, rounds: int = ROUNDS):
    """One group's fp16 table [64] and its weights' indices (uint8, flattened)."""
    v = np.asarray(values, dtype=np.float64).ravel()
    c = initial_table(v)
    for _ in range(rounds):
        c = kmeans_round(v, c)
    table = c.astype(np.float16)
    return table, assign(v, table.astype(np.float64)).astype(np.uint8)


def quantize(w: np.ndarray, rounds: int = ROUNDS):
    """w [n, k] fp16 (n % 16 == 0, k % 4 == 0) -> (packed [n, k*3/4] uint8, lut [n/16, 64] fp16)."""
    w = np.asarray(w, dtype=np.float16)
    n, k = w.shape
    if n % GROUP_ROWS or k % 4 or k == 0:
        raise ValueError("n must be a multiple of 16 and k a positive multiple of 4")
    if not np.isfinite(w).all():
        raise ValueError("weights must be finite")
    idx = np.empty((n, k), dtype=np.uint8)
    lut = np.empty((n // GROUP_ROWS, TABLE_SIZE), dtype=np.float16)
    for g in range(n // GROUP_ROWS):
        rows = slice(GROUP_ROWS * g, GROUP_ROWS * (g + 1))
        table, ind = quantize_group(w[rows].astype(np.float64), rounds)
        lut[g] = table
        idx[rows] = ind.reshape(GROUP_ROWS, k)
    return pack(idx), lut

"""LUT-6 quantiser, oracle side: thin marshalling over the C++ oracle (oracle/csrc/quantize.cpp,
which states the card's method and the readings taken where the card is silent).
"""
from __future__ import annotations

import numpy as np

from ._lib import check, f16_bits, f64, lib, ptr
from .lut6 import GROUP_ROWS, TABLE_SIZE

ROUNDS = 40
HALF = TABLE_SIZE // 2   # quantile seeds, and evenly spread seeds


def quantiles(values: np.ndarray) -> np.ndarray:
    """The 32 quantile seeds of one group, float64 ascending."""
    v = f64(values).ravel()
    out = np.empty(HALF)
    lib().orc_quant_quantiles(ptr(v), v.size, ptr(out))
    return out


def spread(values: np.ndarray) -> np.ndarray:
    """The 32 evenly spread seeds from min to max, float64."""
    v = f64(values).ravel()
    out = np.empty(HALF)
    lib().orc_quant_spread(ptr(v), v.size, ptr(out))
    return out


def initial_table(values: np.ndarray) -> np.ndarray:
    """64 starting centroids of one group (float64, ascending)."""
    v = f64(values).ravel()
    out = np.empty(TABLE_SIZE)
    lib().orc_quant_initial_table(ptr(v), v.size, ptr(out))
    return out


def assign(values: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """Nearest of ascending centroids (ties to the lower index, the first of equal centroids)."""
    v = f64(values).ravel()
    c = f64(centroids).ravel()
    out = np.empty(v.size, dtype=np.int64)
    lib().orc_quant_assign(ptr(v), v.size, ptr(c), c.size, ptr(out))
    return out


def kmeans_round(values: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """One round: assign, move each centroid with members to their mean, sort (stable)."""
    v = f64(values).ravel()
    c = np.array(centroids, dtype=np.float64).ravel()
    lib().orc_quant_kmeans_round(ptr(v), v.size, ptr(c), c.size)
    return c


def quantize_group(values: np.ndarray, rounds: int = ROUNDS):
    """One group's fp16 table [64] and its weights' indices (uint8, flattened)."""
    v = f64(values).ravel()
    table = np.empty(TABLE_SIZE, dtype=np.uint16)
    idx = np.empty(v.size, dtype=np.uint8)
    lib().orc_quant_group(ptr(v), v.size, rounds, ptr(table), ptr(idx))
    return table.view(np.float16), idx


def quantize(w: np.ndarray, rounds: int = ROUNDS):
    """w [n, k] fp16 (n % 16 == 0, k % 4 == 0) -> (packed [n, k*3/4] uint8, lut [n/16, 64] fp16)."""
    bits = f16_bits(w)
    n, k = bits.shape
    if n % GROUP_ROWS or k % 4 or k == 0:
        raise ValueError("n must be a multiple of 16 and k a positive multiple of 4")
    packed = np.empty((n, k * 3 // 4), dtype=np.uint8)
    lut = np.empty((n // GROUP_ROWS, TABLE_SIZE), dtype=np.uint16)
    check(lib().orc_lut6_quantize(ptr(bits), n, k, rounds, ptr(packed), ptr(lut)), "quantize")
    return packed, lut.view(np.float16)

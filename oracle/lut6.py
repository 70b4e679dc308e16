"""LUT-6 weight format, oracle side: thin marshalling over the C++ oracle (oracle/csrc/lut6.cpp).

Source: "Clef-Flash-ANE-LUT6" model card, Weight precision and LUT-6 text weights: a 6-bit index
per weight and one 64-entry FP16 table per 16 output channels, four indices in three bytes in the
little-endian order Core ML uses (read as one LSB-first bit stream over W row-major, k fastest:
w = i0 | i1 << 6 | i2 << 12 | i3 << 18, bytes w & 255, (w >> 8) & 255, w >> 16).  The byte order
is parity unpinned against any external artefact (no page prints one); the round trip and the
hand-worked bytes of (1, 2, 3, 4) -> 81 30 10 pin this reading.
"""
from __future__ import annotations

import numpy as np

from ._lib import check, contig, f16_bits, f64, lib, ptr

GROUP_ROWS = 16      # output channels sharing one table
TABLE_SIZE = 64      # entries per table (6-bit indices)


def pack(idx: np.ndarray) -> np.ndarray:
    """[n, k] uint8 indices (< 64, k % 4 == 0) -> [n, k*3/4] packed bytes."""
    idx = np.asarray(idx)
    n, k = idx.shape
    if k % 4:
        raise ValueError("k must be a multiple of 4")
    if idx.size and (int(idx.min()) < 0 or int(idx.max()) >= TABLE_SIZE):
        raise ValueError("indices must be in 0 .. 63")
    src = contig(idx, np.uint8)
    out = np.empty((n, k * 3 // 4), dtype=np.uint8)
    check(lib().orc_lut6_pack(ptr(src), n, k, ptr(out)), "pack")
    return out


def unpack(packed: np.ndarray, k: int) -> np.ndarray:
    """[n, k*3/4] packed bytes -> [n, k] uint8 indices (inverse of :func:`pack`)."""
    packed = contig(packed, np.uint8)
    n = packed.shape[0]
    if k % 4 or packed.shape[1] != k * 3 // 4:
        raise ValueError("packed row length must be k*3/4 with k % 4 == 0")
    out = np.empty((n, k), dtype=np.uint8)
    check(lib().orc_lut6_unpack(ptr(packed), n, k, ptr(out)), "unpack")
    return out


def _check_lut(lut, n, k, packed):
    if n % GROUP_ROWS or np.shape(lut) != (n // GROUP_ROWS, TABLE_SIZE):
        raise ValueError("lut must be [n/16, 64] with n % 16 == 0")
    if np.shape(packed) != (n, k * 3 // 4):
        raise ValueError("packed must be [n, k*3/4]")


def dequant(packed: np.ndarray, lut: np.ndarray, n: int, k: int) -> np.ndarray:
    """W[r, c] = table[r // 16][idx[r, c]] as float64 [n, k] (exact: fp16 values widen exactly)."""
    _check_lut(lut, n, k, packed)
    p, t = contig(packed, np.uint8), f16_bits(lut)
    out = np.empty((n, k))
    check(lib().orc_lut6_dequant(ptr(p), ptr(t), n, k, ptr(out)), "dequant")
    return out


def dequant_f16(packed: np.ndarray, lut: np.ndarray, n: int, k: int) -> np.ndarray:
    """The same weights kept as fp16 (for bit-exact comparisons)."""
    _check_lut(lut, n, k, packed)
    p, t = contig(packed, np.uint8), f16_bits(lut)
    out = np.empty((n, k), dtype=np.uint16)
    check(lib().orc_lut6_dequant_f16(ptr(p), ptr(t), n, k, ptr(out)), "dequant_f16")
    return out.view(np.float16)


def linear(x: np.ndarray, packed: np.ndarray, lut: np.ndarray, n: int) -> np.ndarray:
    """y = x @ W^T for a LUT-6 weight W [n, k]; x [m, k] (any float), result float64 [m, n]."""
    xx = f64(x)
    m, k = xx.shape
    _check_lut(lut, n, k, packed)
    p, t = contig(packed, np.uint8), f16_bits(lut)
    out = np.empty((m, n))
    check(lib().orc_lut6_linear(ptr(xx), m, k, ptr(p), ptr(t), n, ptr(out)), "linear")
    return out


def storage_bits(n: int, k: int) -> int:
    """Bits stored for an n x k LUT-6 layer: 6 per weight plus 64 fp16 entries per 16 rows."""
    return int(lib().orc_lut6_storage_bits(n, k))


def bits_per_weight(n: int, k: int) -> float:
    return storage_bits(n, k) / (n * k)

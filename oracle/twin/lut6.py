"""LUT-6 weight format: the numpy twin of the C++ oracle (integer work exact, products in float64).

Source: "Clef-Flash-ANE-LUT6" model card, §Weight precision and §LUT-6 text weights:
each large linear stores a 6-bit index per weight and an fp16 table of 64 values for each block
of 16 output channels, 4 indices to 3 bytes in the little-endian order Core ML uses; tables included,
a layer with 4,096 inputs comes to about 6.02 bits per weight.

Reading of "little-endian" (the page gives no byte dump): the indices form one LSB-first bit
stream over the weight matrix in row-major order (input index k fastest).  Indices i0..i3 of a
quadruple make the 24-bit word  w = i0 | i1 << 6 | i2 << 12 | i3 << 18,  stored as the bytes
w & 255, (w >> 8) & 255, w >> 16.  With k a multiple of 4, rows never share a byte.
The byte order is parity unpinned against any external artefact (no page prints one); the
round trip and the hand-worked bytes of (1, 2, 3, 4) -> 81 30 10 pin this reading.
"""
from __future__ import annotations

import numpy as np

GROUP_ROWS = 16      # output channels sharing one table
TABLE_SIZE = 64      # entries per table (6-bit indices)


def pack(idx: np.ndarray) -> np.ndarray:
    """[n, k] uint8 indices (< 64, k % 4 == 0) -> [n, k*3/4] packed bytes."""
    idx = np.asarray(idx)
    n, k = idx.shape
    if k % 4:
        raise ValueError("k must be a multiple of 4")
    if idx.size and int(idx.max()) >= TABLE_SIZE:
        raise ValueError("indices must be below 64")
    q = idx.reshape(n, k // 4, 4).astype(np.uint32)
    w = q[..., 0] | (q[..., 1] << 6) | (q[..., 2] << 12) | (q[..., 3] << 18)
    out = np.empty((n, k // 4, 3), dtype=np.uint8)
    out[..., 0] = w & 0xFF
    out[..., 1] = (w >> 8) & 0xFF
    out[..., 2] = (w >> 16) & 0xFF
    return out.reshape(n, k * 3 // 4)


def unpack(packed: np.ndarray, k: int) -> np.ndarray:
    """[n, k*3/4] packed bytes -> [n, k] uint8 indices (inverse of :func:`pack`)."""
    packed = np.asarray(packed, dtype=np.uint8)
    n = packed.shape[0]
    if k % 4 or packed.shape[1] != k * 3 // 4:
        raise ValueError("packed row length must be k*3/4 with k % 4 == 0")
    # index j is bits 6j .. 6j + 5 of the word w = b0 | b1 << 8 | b2 << 16, read byte by byte
    b = packed.reshape(n, k // 4, 3)
    b0, b1, b2 = b[..., 0], b[..., 1], b[..., 2]
    out = np.empty((n, k // 4, 4), dtype=np.uint8)
    out[..., 0] = b0 & 0x3F
    out[..., 1] = (b0 >> 6) | ((b1 & 0x0F) << 2)
    out[..., 2] = (b1 >> 4) | ((b2 & 0x03) << 4)
    out[..., 3] = b2 >> 2
    return out.reshape(n, k)


def dequant(packed: np.ndarray, lut: np.ndarray, n: int, k: int) -> np.ndarray:
    """W[r, c] = table[r // 16][idx[r, c]] as float64 [n, k] (exact: fp16 values widen exactly)."""
    lut = np.asarray(lut)
    if n % GROUP_ROWS or lut.shape != (n // GROUP_ROWS, TABLE_SIZE):
        raise ValueError("lut must be [n/16, 64] with n % 16 == 0")
    idx = unpack(packed, k)
    table = lut.astype(np.float64)
    out = np.empty((n, k))
    for g in range(n // GROUP_ROWS):
        rows = slice(GROUP_ROWS * g, GROUP_ROWS * (g + 1))
        # table[g][idx[rows]]; 6-bit indices never reach the clip
        np.take(table[g], idx[rows], out=out[rows], mode="clip")
    return out


def dequant_f16(packed: np.ndarray, lut: np.ndarray, n: int, k: int) -> np.ndarray:
    """The same weights kept as fp16 bit patterns (for bit-exact comparisons)."""
    idx = unpack(packed, k)
    group = (np.arange(n) // GROUP_ROWS)[:, None]
    return np.asarray(lut, dtype=np.float16)[group, idx]


def linear(x: np.ndarray, packed: np.ndarray, lut: np.ndarray, n: int) -> np.ndarray:
    """y = x @ W^T for a LUT-6 weight W [n, k]; x [m, k] (any float), result float64 [m, n]."""
    x = np.asarray(x, dtype=np.float64)
    k = x.shape[1]
    return x @ dequant(packed, lut, n, k).T


def storage_bits(n: int, k: int) -> int:
    """Bits stored for an n x k LUT-6 layer: 6 per weight plus 64 fp16 entries per 16 rows."""
    packed_bytes = n * (k * 3 // 4)
    table_bytes = (n // GROUP_ROWS) * TABLE_SIZE * 2
    return 8 * (packed_bytes + table_bytes)


def bits_per_weight(n: int, k: int) -> float:
    return storage_bits(n, k) / (n * k)

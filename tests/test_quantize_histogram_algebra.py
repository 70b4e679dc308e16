"""The LUT-6 quantiser's histogram algorithm equals the oracle's k-means (CPU, exact).

The CUDA quantiser never iterates over a group's weights during k-means: every fp16 bit pattern
maps to a 16-bit key ordered like its value, the group is summarised by counts per key, and each
step of the method becomes lookups in prefix counts and exact integer prefix sums:
  * order statistics (for the quantile seeds): the key at which the prefix count passes a rank;
  * a round: with ascending centroids, the cell of centroid j is the key range from the first key
    above the midpoint below it to the first key above the midpoint above it; its count and sum
    are differences of prefixes; the first key above a midpoint comes from the midpoint's bits
    with integer operations only (its significand cut to fp16 precision);
  * final indices: the number of thresholds at or below the weight's key, mapped to the first of
    any run of equal table entries.
This test writes that algorithm out in numpy (sharing no code with the kernel or the oracle) and
checks that it reproduces the oracle's tables and indices bit for bit ("Clef-Flash-ANE-LUT6"
model card, section "LUT-6 text weights").
"""
import struct

import numpy as np
import pytest

from oracle import quantize as Q

FIX = 2 ** 24


def key_of(h):
    h = np.asarray(h, dtype=np.int64)
    return np.where(h & 0x8000, 0xFFFF - h, h + 0x8000)


def bits_of(key):
    key = np.asarray(key, dtype=np.int64)
    return np.where(key >= 0x8000, key - 0x8000, 0xFFFF - key)


def key_fixed(key):
    """Value in units of 2^-24 (exact for every finite fp16)."""
    h = bits_of(key)
    e, m = (h >> 10) & 31, h & 1023
    mag = np.where(e > 0, (1024 | m) << np.maximum(e - 1, 0), m)
    return np.where(h & 0x8000, -mag, mag)


def key_value(key):
    return float(np.uint16(bits_of(key)).view(np.float16))


def first_key_above(b):
    """The first key whose value is above b, from b's bits with integer operations only."""
    bits = struct.unpack("<Q", struct.pack("<d", b))[0]
    m52, ebits = bits & ((1 << 52) - 1), (bits >> 52) & 0x7FF
    if ebits == 0 and m52 == 0:
        return 0x8001
    E = ebits - 1023
    if E >= -14:
        t, exact = ((E + 15) << 10) | (m52 >> 42), (m52 & ((1 << 42) - 1)) == 0
    else:
        sig, shift = (1 << 52) | m52, 28 - E
        t, exact = (sig >> shift, (sig & ((1 << shift) - 1)) == 0) if shift < 64 else (0, False)
    if not bits >> 63:
        return t + 0x8000 + 1
    if t == 0:
        return 0x7FFF
    k = 0xFFFF - (0x8000 | t)
    return k + 1 if exact else k


def histogram_quantize_group(values16):
    keys = key_of(np.asarray(values16, dtype=np.float16).view(np.uint16).astype(np.int64))
    counts = np.bincount(keys, minlength=65536).astype(np.int64)
    pc = np.concatenate([[0], np.cumsum(counts)])                            # count below key
    ps = np.concatenate([[0], np.cumsum(counts * key_fixed(np.arange(65536)))])   # exact sums
    n = int(pc[-1])

    def at_rank(r):                        # the key holding the r-th smallest weight
        return key_value(int(np.searchsorted(pc, r, side="right")) - 1)

    quant = []
    for i in range(32):
        num = (n - 1) * (2 * i + 1)
        a, b = at_rank(num >> 6), at_rank(min((num >> 6) + 1, n - 1))
        quant.append(a + ((num & 63) / 64.0) * (b - a))
    lo, hi = at_rank(0), at_rank(n - 1)
    step = (hi - lo) / 31
    seeds = quant + [i * step + lo for i in range(31)] + [hi]
    c = [seeds[j] for j in sorted(range(64), key=lambda j: (seeds[j], j))]
    for _ in range(Q.ROUNDS):
        u = [0] + [first_key_above((c[j] + c[j + 1]) * 0.5) for j in range(63)] + [65536]
        new = list(c)
        for j in range(64):
            if j > 0 and c[j - 1] == c[j]:
                continue                   # a run of equal centroids: its first takes the cells
            e = j
            while e < 63 and c[e + 1] == c[j]:
                e += 1
            cnt = int(pc[u[e + 1]] - pc[u[j]])
            if cnt:
                new[j] = (float(int(ps[u[e + 1]] - ps[u[j]])) / cnt) / FIX
        c = [new[j] for j in sorted(range(64), key=lambda j: (new[j], j))]
    table = np.array(c).astype(np.float16)
    t64 = table.astype(np.float64)
    thr = np.array([first_key_above((t64[j] + t64[j + 1]) * 0.5) for j in range(63)])
    first = np.array([min(i for i in range(64) if t64[i] == t64[j]) for j in range(64)])
    cell = np.searchsorted(thr, keys, side="right")    # thresholds at or below the key
    return table, first[cell].astype(np.uint8)


def _group(kind, seed):
    rng = np.random.default_rng(seed)
    n = 16 * 96
    if kind == "normal":
        v = rng.standard_normal(n) * 0.02
    elif kind == "heavy":
        v = rng.standard_t(2.5, n) * 0.02
    elif kind == "wide":
        v = rng.standard_normal(n) * rng.choice([0.01, 1.0, 50.0], n)
    elif kind == "levels":
        v = rng.choice([-0.5, -0.125, 0.0, 0.25, 3.0], n)
    else:                                  # subnormals and zeros of both signs
        v = rng.standard_normal(n) * 2e-6
        v[::7], v[::11] = -0.0, 0.0
    return v.astype(np.float16)


@pytest.mark.parametrize("kind", ["normal", "heavy", "wide", "levels", "tiny"])
@pytest.mark.parametrize("seed", [0, 1])
def test_histogram_algorithm_equals_oracle(kind, seed):
    v = _group(kind, seed)
    table, idx = histogram_quantize_group(v)
    ref_table, ref_idx = Q.quantize_group(v.astype(np.float64))
    assert np.array_equal(table.view(np.uint16), ref_table.view(np.uint16))
    assert np.array_equal(idx, ref_idx)


def test_block_linear_values():
    """Inside a 32-key block (never across an fp16 binade) the value is linear in the key: the
    kernel's in-block partial sums use f0 * count + step * first moment."""
    for key0 in range(0, 65536, 32):
        h = int(bits_of(key0))
        e = (h >> 10) & 31
        if e == 31:
            continue
        step = (1 << (e - 1)) if e >= 2 else 1
        ks = np.arange(key0, key0 + 32)
        assert np.array_equal(key_fixed(ks), key_fixed(key0) + np.arange(32) * step)


def test_first_key_above_on_all_fp16_values_and_midpoints():
    f = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (f[:-1] + f[1:]) / 2
    for b in np.concatenate([f[1::97], -f[1::97], mids[::89], -mids[::89]]):
        k = first_key_above(float(b))
        assert key_value(k) > b                               # above b ...
        assert key_value(k - 1) <= b or k - 1 == 0x7FFF and b < 0  # ... and the first one

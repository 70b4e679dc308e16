"""Pins of the LUT-6 quantiser oracle (CPU).

"Clef-Flash-ANE-LUT6" model card, section "LUT-6 text weights": a 64-entry table per 16 output
channels, 40 k-means iterations in one dimension, initial centroids 32 quantiles and 32 equal
steps from the smallest to the largest weight.  The oracle is pinned to things outside itself: numpy's
own quantile and linspace, exact rational arithmetic (Python fractions) for nearest centroids,
means and a whole brute-force k-means on small groups, special cases with known answers, the
k-means descent invariant, and the Panter-Dite high-resolution distortion of a Gaussian source.
"""
from fractions import Fraction
import math

import numpy as np
import pytest

from oracle import lut6
from oracle import quantize as Q


def _fp16(rng, n, scale=0.02):
    return (rng.standard_normal(n) * scale).astype(np.float16).astype(np.float64)


@pytest.mark.parametrize("n", [64, 65, 1000, 4096, 16 * 768])
def test_quantile_seeds_equal_numpy_quantile(n):
    rng = np.random.default_rng(n)
    v = _fp16(rng, n)
    probs = (np.arange(32) + 0.5) / 32
    assert np.array_equal(Q.quantiles(v), np.quantile(v, probs))        # default: linear


def test_quantile_seeds_are_exact():
    """Every step is exact for fp16 data: compare with rational arithmetic."""
    rng = np.random.default_rng(1)
    v = _fp16(rng, 777, scale=3.0)
    x = sorted(Fraction(float(t)) for t in v)
    n = len(x)
    for i, q in enumerate(Q.quantiles(v)):
        h = Fraction(2 * i + 1, 64) * (n - 1)
        lo = math.floor(h)
        exact = x[lo] + (h - lo) * (x[min(lo + 1, n - 1)] - x[lo])
        assert Fraction(float(q)) == exact


def test_quantiles_of_an_arithmetic_sequence():
    """For the values 0..n-1 the interpolated quantile is the fractional rank itself."""
    n = 64
    v = np.arange(n, dtype=np.float64)
    expect = (np.arange(32) + 0.5) / 32 * (n - 1)
    assert np.array_equal(Q.quantiles(v), expect)
    assert Q.quantiles(v)[0] == 63 / 64 and Q.quantiles(v)[31] == 63 - 63 / 64


@pytest.mark.parametrize("seed", range(6))
def test_spread_seeds_equal_numpy_linspace(seed):
    rng = np.random.default_rng(100 + seed)
    v = _fp16(rng, 200, scale=[1e-3, 0.02, 1.0, 30.0, 1e4, 0.0][seed])
    s = Q.spread(v)
    assert np.array_equal(s, np.linspace(v.min(), v.max(), 32))
    assert s[0] == v.min() and s[-1] == v.max()
    assert np.all(np.diff(s) >= 0)


def test_initial_table_is_the_two_halves_sorted():
    rng = np.random.default_rng(2)
    v = _fp16(rng, 16 * 64)
    t = Q.initial_table(v)
    assert t.shape == (64,) and np.all(np.diff(t) >= 0)
    assert sorted(t.tolist()) == sorted(Q.quantiles(v).tolist() + Q.spread(v).tolist())
    assert t[0] == v.min() and t[-1] == v.max()


def _nearest_exact(values, centroids):
    """Brute force: exact distances in rationals, first minimum (lowest index) wins."""
    cs = [Fraction(float(c)) for c in centroids]
    out = []
    for v in values:
        fv = Fraction(float(v))
        d = [abs(fv - c) for c in cs]
        out.append(d.index(min(d)))
    return np.array(out)


def test_assign_is_nearest_with_ties_to_lower_index():
    rng = np.random.default_rng(3)
    c = np.sort(_fp16(rng, 64, scale=0.05))
    v = _fp16(rng, 2000, scale=0.06)
    # weights lying exactly on midpoints of fp16 centroids go to the lower index
    mids = ((c[:-1] + c[1:]) / 2).astype(np.float16).astype(np.float64)
    on_mid = mids[(mids * 2 == c[:-1] + c[1:])]
    v = np.concatenate([v, on_mid, c])
    assert on_mid.size > 5
    got = Q.assign(v, c)
    assert np.array_equal(got, _nearest_exact(v, c))


def test_assign_with_repeated_centroids():
    c = np.array([0.0, 0.0, 1.0, 1.0, 1.0, 2.0])
    v = np.array([-1.0, 0.0, 0.4, 0.5, 0.6, 1.0, 1.5, 1.6, 3.0])
    assert Q.assign(v, c).tolist() == _nearest_exact(v, c).tolist() == [0, 0, 0, 0, 2, 2, 2, 5, 5]


def test_round_means_are_the_correctly_rounded_rational_means():
    rng = np.random.default_rng(4)
    v = _fp16(rng, 3000)
    c0 = Q.initial_table(v)
    c1 = Q.kmeans_round(v, c0)
    a = _nearest_exact(v, c0)
    expect = []
    for j in range(64):
        members = [Fraction(float(t)) for t in v[a == j]]
        expect.append(float(sum(members) / len(members)) if members else c0[j])
    assert np.array_equal(c1, np.sort(expect))


def _kmeans_brute(values, rounds):
    """The card's k-means in rationals: exact nearest, exact mean rounded once to float64, the
    centroids kept in ascending order (stable)."""
    c = [float(t) for t in Q.initial_table(values)]
    vals = [Fraction(float(t)) for t in values]
    for _ in range(rounds):
        a = _nearest_exact(values, c)
        for j in range(len(c)):
            members = [vals[i] for i in range(len(vals)) if a[i] == j]
            if members:
                c[j] = float(sum(members) / len(members))
        c = [c[j] for j in sorted(range(len(c)), key=lambda j: c[j])]   # Python's sort is stable
    table = np.array(c).astype(np.float16)
    return table, _nearest_exact(values, table.astype(np.float64))


@pytest.mark.parametrize("seed", range(3))
def test_quantize_group_matches_rational_brute_force(seed):
    rng = np.random.default_rng(10 + seed)
    v = _fp16(rng, 16 * 8, scale=[0.02, 1.0, 300.0][seed])
    table, idx = Q.quantize_group(v)
    bt, bidx = _kmeans_brute(v, Q.ROUNDS)
    assert np.array_equal(table.view(np.uint16), bt.view(np.uint16))
    assert np.array_equal(idx, bidx)


def test_repeated_seeds_match_rational_brute_force():
    """Many equal quantile seeds (a few values repeated, zeros of both signs): the case where the
    first of several equal centroids moves alone."""
    rng = np.random.default_rng(21)
    v = rng.choice(np.array([-0.0, 0.0, 2.0 ** -24, 3 * 2.0 ** -24, -2.0 ** -23, 0.5]), size=16 * 8)
    v = np.concatenate([v, _fp16(rng, 16 * 4, 1e-6)])
    table, idx = Q.quantize_group(v)
    bt, bidx = _kmeans_brute(v, Q.ROUNDS)
    assert np.array_equal(table.view(np.uint16), bt.view(np.uint16))
    assert np.array_equal(idx, bidx)
    assert np.all(np.diff(table.astype(np.float64)) >= 0)


def test_constant_group():
    v = np.full(16 * 8, 0.375)
    table, idx = Q.quantize_group(v)
    assert np.all(table == np.float16(0.375)) and np.all(idx == 0)


@pytest.mark.parametrize("levels", [1, 2, 7, 32])
def test_few_equally_frequent_levels_are_reproduced_exactly(levels):
    """Every level then holds a quantile seed, so it keeps a centroid of its own."""
    rng = np.random.default_rng(levels)
    vals = np.sort(_fp16(rng, levels, scale=0.5))
    vals = np.unique(vals)
    per = (16 * 64) // vals.size
    v = rng.permutation(np.repeat(vals, per))[: 16 * (per * vals.size // 16)]
    table, idx = Q.quantize_group(v)
    assert np.array_equal(table.astype(np.float64)[idx], v)


def test_centroids_stay_ascending_and_objective_descends():
    rng = np.random.default_rng(5)
    v = np.concatenate([_fp16(rng, 16 * 200, 0.01), _fp16(rng, 16 * 56, 0.2) + 0.5])
    c = Q.initial_table(v)
    prev = np.inf
    for _ in range(Q.ROUNDS):
        c = Q.kmeans_round(v, c)
        assert np.all(np.diff(c) >= 0)
        sse = float(np.sum((v - c[Q.assign(v, c)]) ** 2))
        assert sse <= prev * (1 + 1e-12)
        prev = sse


def test_gaussian_distortion_near_panter_dite():
    """High-resolution theory: a 64-level optimal quantiser of a Gaussian leaves an MSE of
    about (sqrt(3) pi / 2) sigma^2 / 64^2 (Panter and Dite, 1951)."""
    rng = np.random.default_rng(6)
    sigma = 0.02
    v = _fp16(rng, 16 * 1024, sigma)
    table, idx = Q.quantize_group(v)
    mse = float(np.mean((v - table.astype(np.float64)[idx]) ** 2))
    pd = math.sqrt(3) * math.pi / 2 * np.var(v) / 64 ** 2
    assert 0.75 * pd < mse < 1.15 * pd


def test_final_indices_are_nearest_table_entries_and_roundtrip():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((32, 64)) * 0.03).astype(np.float16)
    packed, lut = Q.quantize(w)
    assert packed.shape == (32, 48) and lut.shape == (2, 64) and lut.dtype == np.float16
    idx = lut6.unpack(packed, 64)
    for g in range(2):
        rows = slice(16 * g, 16 * g + 16)
        vals = w[rows].astype(np.float64).ravel()
        assert np.array_equal(idx[rows].ravel(), _nearest_exact(vals, lut[g].astype(np.float64)))
        assert np.all(np.diff(lut[g].astype(np.float64)) >= 0)
    deq = lut6.dequant(packed, lut, 32, 64)
    rel = np.sqrt(np.mean((deq - w) ** 2) / np.mean(w.astype(np.float64) ** 2))
    assert rel < 0.05


def test_quantize_rejects_bad_input():
    with pytest.raises(ValueError):
        Q.quantize(np.zeros((15, 8), np.float16))
    with pytest.raises(ValueError):
        Q.quantize(np.zeros((16, 6), np.float16))
    w = np.zeros((16, 8), np.float16)
    w[3, 3] = np.inf
    with pytest.raises(ValueError):
        Q.quantize(w)

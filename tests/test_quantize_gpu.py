"""LUT-6 quantiser on the GPU against the oracle (bit-exact indices and tables).

Both sides follow one exactly specified arithmetic (exact integer sums, one rounding per mean,
fp16 rounding of the final table), so the packed bytes and the tables must agree bit for bit.
Cases: typical weights (normal, std 0.02), heavy tails reaching the outer key quarters, values
spanning all four quarters, constant and few-level groups, signed zeros and subnormals, a ragged
k (not a multiple of 8), more groups than resident clusters (persistent walk), and a full-size
4096 x 4096 weight checked on sampled groups plus properties of every group.
"""
import numpy as np
import pytest

import synth
from oracle import lut6 as olut
from oracle import quantize as oq

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402


def _quantize(w):
    packed, lut = clef.lut6_quantize(torch.from_numpy(np.ascontiguousarray(w)).cuda())
    clef.sync_status()
    return packed.cpu().numpy(), lut.cpu().numpy()


def _assert_same(w):
    packed, lut = _quantize(w)
    rp, rl = oq.quantize(w)
    assert np.array_equal(lut.view(np.uint16), rl.view(np.uint16))
    assert np.array_equal(packed, rp)


def _weights(kind, n, k, seed=0):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return synth.normal_f16(seed, "qw", 0, (n, k), std=0.02)
    if kind == "heavy":          # Student-t tails: a few weights far outside the bulk
        return (rng.standard_t(2.5, size=(n, k)) * 0.02).astype(np.float16)
    if kind == "wide":           # every key quarter: |w| above and below 2, both signs
        return (rng.standard_normal((n, k)) * rng.choice([0.01, 1.0, 50.0], size=(n, k))).astype(np.float16)
    if kind == "levels":         # few distinct values per group, some groups constant
        w = rng.choice(np.array([-0.5, -0.125, 0.0, 0.25, 3.0], np.float16), size=(n, k))
        w[:16] = np.float16(0.375)
        return w
    if kind == "tiny":           # subnormals and both signed zeros
        w = (rng.standard_normal((n, k)) * 2e-6).astype(np.float16)
        w[:, ::7] = np.float16(-0.0)
        w[:, ::11] = np.float16(0.0)
        w[16:32] = np.float16(-0.0)     # a group of negative zeros only
        return w
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "heavy", "wide", "levels", "tiny"])
def test_bit_exact_small(kind):
    _assert_same(_weights(kind, 64, 256, seed=len(kind)))


@pytest.mark.parametrize("n,k", [(16, 4), (32, 1028), (48, 12)])
def test_bit_exact_ragged_shapes(n, k):
    _assert_same(_weights("normal", n, k, seed=n + k))


def test_bit_exact_more_groups_than_clusters():
    # 116 groups: more than the clusters resident at once, so clusters take several groups
    _assert_same(_weights("heavy", 16 * 116, 64, seed=3))


def test_dequant_roundtrip_and_status():
    w = _weights("normal", 64, 512, seed=9)
    packed, lut = clef.lut6_quantize(torch.from_numpy(w).cuda())
    deq = clef.lut6_dequant(packed, lut, 512)
    clef.sync_status()
    idx = olut.unpack(packed.cpu().numpy(), 512)
    group = (np.arange(64) // 16)[:, None]
    assert np.array_equal(deq.cpu().numpy().view(np.uint16), lut.cpu().numpy()[group, idx].view(np.uint16))


def test_nonfinite_is_reported():
    w = _weights("normal", 32, 64, seed=4)
    w[20, 5] = np.float16(np.inf)
    packed, lut = clef.lut6_quantize(torch.from_numpy(w).cuda())
    with pytest.raises(clef.ClefError) as e:
        clef.sync_status()
    assert e.value.code == 7
    clef.sync_status()            # the status word is cleared after the report


def test_shape_errors():
    with pytest.raises(clef.ClefError) as e:
        clef.lut6_quantize(torch.zeros((24, 8), dtype=torch.float16, device="cuda"))
    assert e.value.code == 2
    with pytest.raises(clef.ClefError) as e:
        clef.lut6_quantize(torch.zeros((16, 6), dtype=torch.float16, device="cuda"))
    assert e.value.code == 2


@pytest.mark.slow
def test_full_size_4096x4096():
    n = k = 4096
    w = _weights("normal", n, k, seed=11)
    packed, lut = _quantize(w)
    assert np.all(np.diff(lut.astype(np.float64), axis=1) >= 0)
    # sampled groups against the oracle, bit for bit
    for g in (0, 97, 255):
        rows = slice(16 * g, 16 * g + 16)
        table, ind = oq.quantize_group(w[rows].astype(np.float64))
        assert np.array_equal(lut[g].view(np.uint16), table.view(np.uint16))
        assert np.array_equal(olut.unpack(packed[rows], k).ravel(), ind)
    # every group: each index is a nearest entry of its own table
    idx = torch.from_numpy(olut.unpack(packed, k).astype(np.int64)).cuda()
    t = torch.from_numpy(lut.astype(np.float64)).cuda()          # differences exact in fp64
    wv = torch.from_numpy(w.astype(np.float64)).cuda()
    grp = (torch.arange(n, device="cuda") // 16)[:, None]
    got = (wv - t[grp, idx]).abs()
    best = torch.full_like(got, float("inf"))
    for j in range(64):
        best = torch.minimum(best, (wv - t[grp.expand(n, k), torch.full_like(idx, j)]).abs())
    assert torch.equal(got, best)
    rel = float(((wv - t[grp, idx]) ** 2).mean().sqrt() / (wv ** 2).mean().sqrt())
    print(f"4096 x 4096 LUT-6: relative RMS error {rel:.4f}")
    assert rel < 0.04

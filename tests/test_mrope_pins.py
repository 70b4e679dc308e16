"""Pins of the oracle's M-RoPE (CPU): positions of a request with a picture, plane layout, and the
three-plane rotary ("clef-flash-LiteRT" README, "Host contract" step 5; "clef-flash - Core AI"
README, "Core AI shape").
"""
import math
import os

import numpy as np
import pytest

from oracle import layers as Lr
from oracle import model as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mrope_positions_example.txt")


def test_positions_match_hand_worked_example():
    rows = [list(map(int, l.split())) for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    pos = Lr.mrope_positions(46, 37, 2, 3)
    for i, t, h, w in rows:
        assert tuple(pos[i]) == (t, h, w), i


def test_text_only_is_the_ramp():
    pos = Lr.mrope_positions(50)
    assert np.array_equal(pos, np.repeat(np.arange(50)[:, None], 3, axis=1))


@pytest.mark.parametrize("h,w", [(8, 8), (14, 14), (3, 5), (5, 3), (1, 7)])
def test_shift_after_the_picture(h, w):
    """From the <|vision_end|> index 37 + N on, positions move back by N - max(H, W) (the page's
    rope_shift_start / rope_shift_amount), which continues one past the largest picture position."""
    n, s = h * w, 37
    L = s + n + 5
    pos = Lr.mrope_positions(L, s, h, w)
    end = s + n
    assert tuple(pos[end]) == (end - (n - max(h, w)),) * 3
    assert pos[end, 0] == pos[s:end].max() + 1
    # row and column of image token k are k // W and k % W (the page's image_rc)
    k = np.arange(n)
    assert np.array_equal(pos[s:end, 1] - s, k // w) and np.array_equal(pos[s:end, 2] - s, k % w)
    assert np.all(pos[s:end, 0] == s)


def test_planes_interleaved_11_11_10():
    planes = Lr.mrope_planes()
    assert tuple(np.bincount(planes, minlength=3)) == Lr.MROPE_SECTIONS == (11, 11, 10)
    assert planes[:6].tolist() == [0, 1, 2, 0, 1, 2] and planes[31] == 1


def test_mrope_with_equal_planes_is_the_1d_rotary():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((20, 3, 256))
    pos = np.arange(20) * 7 + 3
    assert np.array_equal(Lr.mrope(x, np.repeat(pos[:, None], 3, axis=1)), Lr.rope(x, pos))


@pytest.mark.parametrize("j", [0, 1, 2, 31])
def test_single_pair_closed_form(j):
    """A unit vector in dim j turns by the angle of its plane's position: (cos a, sin a) on dims
    (j, j + 32), a = pos_plane * 10^(-7 j / 32)."""
    pos3 = np.array([[5, 1000, 123456]])
    x = np.zeros((1, 1, 256))
    x[0, 0, j] = 1.0
    y = Lr.mrope(x, pos3)[0, 0]
    a = pos3[0, j % 3] * 10.0 ** (-7.0 * j / 32.0)
    assert y[j] == pytest.approx(math.cos(a), abs=1e-12)
    assert y[j + 32] == pytest.approx(math.sin(a), abs=1e-12)
    assert np.count_nonzero(np.abs(y) > 1e-15) <= 2


def test_only_the_moved_plane_changes_its_pairs():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 2, 256))
    pos3 = Lr.mrope_positions(6, 1, 2, 2)
    for plane in range(3):
        moved = pos3.copy()
        moved[:, plane] += 11
        d = np.abs(Lr.mrope(x, moved) - Lr.mrope(x, pos3)).max(axis=(0, 1))
        pairs = [j for j in range(32) if d[j] > 1e-9 or d[j + 32] > 1e-9]
        assert pairs == [j for j in range(32) if j % 3 == plane]
        assert np.all(d[64:] == 0)


def test_relative_positions_and_norm():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((9, 1, 256))
    k = rng.standard_normal((9, 1, 256))
    pos3 = Lr.mrope_positions(9, 2, 2, 2)
    dots = np.einsum("ld,md->lm", Lr.mrope(q, pos3)[:, 0], Lr.mrope(k, pos3)[:, 0])
    dots2 = np.einsum("ld,md->lm", Lr.mrope(q, pos3 + 100)[:, 0], Lr.mrope(k, pos3 + 100)[:, 0])
    assert np.allclose(dots, dots2, rtol=0, atol=1e-9)
    assert np.allclose(np.linalg.norm(Lr.mrope(q, pos3), axis=-1), np.linalg.norm(q, axis=-1))


def test_attention_mixer_text_positions_as_planes():
    import synth
    w = synth.attention_layer_weights(0, 3)
    xn = synth.normal_f64(0, "mx", 0, (12, 4096))
    a = om.attention_mixer(xn, w)
    b = om.attention_mixer(xn, w, Lr.mrope_positions(12))
    assert np.array_equal(a, b)

"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: the pages' printed figures
(tests/golden/), hand-worked values, closed forms, invariants and brute force on tiny inputs.
"""
import itertools
import math
import os

import numpy as np
import pytest

from oracle import layers as Lr
from oracle import lut6, model

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ------------------------------------------------------------------------------------ LUT-6
def _golden_pack():
    rows = []
    for line in open(os.path.join(GOLDEN, "lut6_pack_examples.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split("|")
        rows.append(([int(t) for t in a.split()], [int(t, 16) for t in b.split()]))
    return rows


def test_pack_hand_worked_bytes():
    rows = _golden_pack()
    assert len(rows) >= 8
    for idx, expect in rows:
        got = lut6.pack(np.array([idx], dtype=np.uint8))
        assert list(got[0]) == expect, (idx, list(got[0]), expect)
        back = lut6.unpack(np.array([expect], dtype=np.uint8), 4)
        assert list(back[0]) == idx


def test_pack_roundtrip_all_quadruples():
    # every one of the 64^4 quadruples, as one row
    q = np.array(np.meshgrid(*[np.arange(64, dtype=np.uint8)] * 4, indexing="ij")).reshape(4, -1).T
    idx = q.reshape(1, -1)
    packed = lut6.pack(idx)
    assert packed.shape == (1, idx.shape[1] * 3 // 4)
    assert np.array_equal(lut6.unpack(packed, idx.shape[1]), idx)
    # the packing is a bijection onto the 2^24 byte triples
    trip = packed.reshape(-1, 3).astype(np.uint32)
    words = trip[:, 0] | (trip[:, 1] << 8) | (trip[:, 2] << 16)
    assert np.unique(words).size == 1 << 24


def _bitstream_weight(packed_row_major: bytes, k: int, r: int, c: int) -> int:
    """Index (r, c) read as bits 6*(r*k+c) .. +5 of one LSB-first stream (independent route)."""
    bit = 6 * (r * k + c)
    v = 0
    for j in range(6):
        byte = packed_row_major[(bit + j) // 8]
        v |= ((byte >> ((bit + j) % 8)) & 1) << j
    return v


def test_unpack_matches_lsb_first_bitstream():
    n, k = 3, 12
    idx = rng.integers(0, 64, size=(n, k), dtype=np.uint8)
    packed = lut6.pack(idx)
    stream = packed.tobytes()
    for r in range(n):
        for c in range(k):
            assert _bitstream_weight(stream, k, r, c) == idx[r, c]


def test_dequant_uses_table_of_row_group():
    n, k = 48, 8
    lut = (np.arange(n // 16 * 64, dtype=np.float64).reshape(n // 16, 64) * 0.25 - 7).astype(np.float16)
    idx = rng.integers(0, 64, size=(n, k), dtype=np.uint8)
    W = lut6.dequant(lut6.pack(idx), lut, n, k)
    for r in range(n):
        for c in range(k):
            assert W[r, c] == float(lut[r // 16, idx[r, c]])


def test_linear_brute_force_tiny():
    m, n, k = 3, 32, 8
    idx = rng.integers(0, 64, size=(n, k), dtype=np.uint8)
    packed = lut6.pack(idx)
    lut = rng.normal(0, 0.5, size=(n // 16, 64)).astype(np.float16)
    x = rng.normal(size=(m, k)).astype(np.float16)
    stream = packed.tobytes()
    y = lut6.linear(x, packed, lut, n)
    for i in range(m):
        for r in range(n):
            s = 0.0
            for c in range(k):
                s += float(x[i, c]) * float(lut[r // 16, _bitstream_weight(stream, k, r, c)])
            assert abs(y[i, r] - s) <= 1e-12 * (1 + abs(s))


def _golden_storage():
    d = {}
    for line in open(os.path.join(GOLDEN, "lut6_storage.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            key, val = line.split()
            d[key] = float(val)
    return d


def test_bits_per_weight_closed_form():
    g = _golden_storage()
    b = lut6.bits_per_weight(4096, 4096)
    assert b == 6 + 1024 / 65536 == 6.015625
    assert round(b, 2) == g["bits_per_weight_k4096"]
    # 6 + 64/k in general (64 fp16 entries per 16 rows)
    for k in (1024, 4096, 12288):
        assert lut6.bits_per_weight(16 * 7, k) == pytest.approx(6 + 64 / k, rel=0, abs=1e-12)


def _lut_layer_shapes(gated_q=True):
    """(n, k) of every LUT-6 linear of the 32-layer backbone."""
    shapes = []
    for layer in range(32):
        if model.is_attention_layer(layer):
            shapes += [(8192 if gated_q else 4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096)]
        else:
            shapes += [(8192, 4096), (4096, 4096), (4096, 4096)]
        shapes += [(12288, 4096), (12288, 4096), (4096, 12288)]
    return shapes


def _small_fp16_weights():
    """Count of the FP16 small text weights (norms, conv, gate projections, decay parameters)."""
    n = 0
    for layer in range(32):
        n += 2 * 4096                                 # two RMSNorms
        if not model.is_attention_layer(layer):
            n += 8192 * 4 + 2 * 32 * 4096 + 2 * 32 + 128
    return n


def test_model_storage_matches_cards_and_pins_gated_query():
    g = _golden_storage()
    for gated, should_match in ((True, True), (False, False)):
        shapes = _lut_layer_shapes(gated)
        lut_bytes = sum(lut6.storage_bits(n, k) for n, k in shapes) // 8
        ane_gib = (lut_bytes + 2 * _small_fp16_weights()) / 2 ** 30
        weights = sum(n * k for n, k in shapes)
        fp16_bytes = 2 * (weights + _small_fp16_weights() + 4096 + 248320 * 4096)
        ok_ane = abs(ane_gib - g["ane_programs_gib"]) < 0.015
        ok_fp16 = abs(fp16_bytes / g["fp16_decoder_bytes"] - 1) < 2e-3
        assert ok_ane == should_match, ane_gib
        assert ok_fp16 == should_match, fp16_bytes
        if gated:
            assert weights == 6_912_212_992


# ----------------------------------------------------------------------------- norms / conv
def test_rmsnorm_constant_row():
    w = rng.normal(1, 0.02, size=64)
    for c in (-3.0, 0.5, 10.0):
        y = Lr.rmsnorm(np.full((1, 64), c), w)
        np.testing.assert_allclose(y[0], w * c / math.sqrt(c * c + 1e-6), rtol=1e-14)


def test_rmsnorm_scale_invariance_and_rms():
    x = rng.normal(size=(5, 256)) * 7
    y = Lr.rmsnorm(x, np.ones(256), eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(Lr.rmsnorm(3 * x, np.ones(256), eps=0.0), y, rtol=1e-13)


def test_l2norm_unit():
    x = rng.normal(size=(4, 3, 128))
    y = Lr.l2norm(x, eps=0.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(y[0, 0] / y[0, 0, 0], x[0, 0] / x[0, 0, 0], rtol=1e-12)


def test_conv_impulse_response():
    L, C = 9, 5
    w = rng.normal(size=(C, 4))
    for t0 in (0, 3, 7):
        x = np.zeros((L, C))
        x[t0, 2] = 1.0
        y = Lr.causal_conv_silu(x, w)
        for t in range(L):
            d = t - t0
            pre = w[2, 3 - d] if 0 <= d <= 3 else 0.0
            assert y[t, 2] == pytest.approx(pre / (1 + math.exp(-pre)), rel=1e-14, abs=1e-300)
            assert np.all(y[t, [0, 1, 3, 4]] == 0.0)


def test_conv_linear_part_against_convolve():
    L, C = 11, 3
    x = rng.normal(size=(L, C))
    w = rng.normal(size=(C, 4))
    y = Lr.causal_conv_silu(x, w)
    for ch in range(C):
        # causal correlation: sum_j w[j] x[t-3+j] == np.convolve with the flipped kernel
        pre = np.convolve(x[:, ch], w[ch, ::-1])[:L]
        np.testing.assert_allclose(y[:, ch], pre / (1 + np.exp(-pre)), rtol=1e-13)


def test_gate_closed_forms():
    A_log = np.array([math.log(0.1), 0.0])
    dt_bias = np.array([0.3, -1.0])
    a = -dt_bias[None, :]                      # softplus(0) = ln 2
    b = np.zeros((1, 2))
    alpha, beta = Lr.gdn_gates(a, b, A_log, dt_bias)
    np.testing.assert_allclose(alpha[0], [2 ** -0.1, 2 ** -1.0], rtol=1e-14)
    np.testing.assert_allclose(beta[0], 0.5, rtol=0)
    # large negative pre-activation: no decay; large positive b: full write
    alpha, beta = Lr.gdn_gates(np.full((1, 2), -800.0), np.full((1, 2), 800.0), A_log, dt_bias)
    np.testing.assert_allclose(alpha, 1.0)
    np.testing.assert_allclose(beta, 1.0)


# ------------------------------------------------------------------------------ delta rule
def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def test_delta_rule_beta0_alpha1_keeps_state():
    L, Hk, Hv, d = 6, 2, 4, 8
    q = rng.normal(size=(L, Hk, d))
    k = _unit(rng.normal(size=(L, Hk, d)))
    v = rng.normal(size=(L, Hv, d))
    s0 = rng.normal(size=(Hv, d, d))
    o, S = Lr.gated_delta_rule(q, k, v, np.ones((L, Hv)), np.zeros((L, Hv)), s0)
    np.testing.assert_array_equal(S, s0)
    qh = np.repeat(q, 2, axis=1)
    np.testing.assert_allclose(o, np.einsum("hij,thj->thi", s0, qh) / math.sqrt(d), rtol=1e-13)


def test_delta_rule_alpha1_beta1_maps_k_to_v():
    L, Hk, Hv, d = 7, 2, 4, 16
    q = rng.normal(size=(L, Hk, d))
    k = _unit(rng.normal(size=(L, Hk, d)))
    v = rng.normal(size=(L, Hv, d))
    s = rng.normal(size=(Hv, d, d))
    for t in range(L):
        _, s = Lr.gated_delta_rule(q[t:t + 1], k[t:t + 1], v[t:t + 1], np.ones((1, Hv)),
                                   np.ones((1, Hv)), s)
        kt = np.repeat(k[t], 2, axis=0)
        np.testing.assert_allclose(np.einsum("hij,hj->hi", s, kt), v[t], atol=1e-12)


def test_delta_rule_alpha0_beta1_is_outer_product():
    L, Hk, Hv, d = 5, 1, 2, 4
    q = rng.normal(size=(L, Hk, d))
    k = _unit(rng.normal(size=(L, Hk, d)))
    v = rng.normal(size=(L, Hv, d))
    o, S = Lr.gated_delta_rule(q, k, v, np.zeros((L, Hv)), np.ones((L, Hv)), rng.normal(size=(Hv, d, d)))
    for h in range(Hv):
        np.testing.assert_allclose(S[h], np.outer(v[-1, h], k[-1, 0]), rtol=1e-14)
        # o_t = v_t (k_t . q_t) / sqrt(d): the output is read after the update
        np.testing.assert_allclose(o[:, h], v[:, h] * np.sum(k[:, 0] * q[:, 0], -1)[:, None] / 2.0,
                                   rtol=1e-13)


def test_delta_rule_scalar_closed_form():
    # d = 1, k = +-1: S_t = alpha_t (1 - beta_t) S_{t-1} + beta_t v_t k_t
    #   => S_L = sum_t beta_t v_t k_t prod_{s>t} alpha_s (1 - beta_s)
    L = 12
    k = rng.choice([-1.0, 1.0], size=(L, 1, 1))
    v = rng.normal(size=(L, 1, 1))
    q = rng.normal(size=(L, 1, 1))
    alpha = rng.uniform(0.3, 1.0, size=(L, 1))
    beta = rng.uniform(0.0, 1.0, size=(L, 1))
    o, S = Lr.gated_delta_rule(q, k, v, alpha, beta)
    decay = alpha[:, 0] * (1 - beta[:, 0])
    expect = sum(beta[t, 0] * v[t, 0, 0] * k[t, 0, 0] * np.prod(decay[t + 1:]) for t in range(L))
    assert S[0, 0, 0] == pytest.approx(expect, rel=1e-12)
    # o_L = S_L q_L (d = 1, scale 1)
    assert o[-1, 0, 0] == pytest.approx(expect * q[-1, 0, 0], rel=1e-12)


def test_delta_rule_head_mapping():
    # value head h reads key head h // 2
    L, Hk, Hv, d = 1, 2, 4, 4
    k = np.zeros((L, Hk, d))
    k[0, 0, 0] = 1.0
    k[0, 1, 1] = 1.0
    v = np.ones((L, Hv, d))
    _, S = Lr.gated_delta_rule(np.zeros((L, Hk, d)), k, v, np.ones((L, Hv)), np.ones((L, Hv)))
    for h in range(Hv):
        col = h // 2
        assert np.all(S[h][:, col] == 1.0) and np.count_nonzero(S[h]) == d


# ------------------------------------------------------------------------------- attention
def test_attention_brute_force_tiny():
    L, Hq, Hkv, D = 6, 4, 2, 3
    q, k, v = rng.normal(size=(L, Hq, D)), rng.normal(size=(L, Hkv, D)), rng.normal(size=(L, Hkv, D))
    o = Lr.causal_attention(q, k, v)
    for h in range(Hq):
        g = h // 2
        for t in range(L):
            logits = [sum(q[t, h, i] * k[s, g, i] for i in range(D)) / math.sqrt(D) for s in range(t + 1)]
            w = [math.exp(z) for z in logits]
            tot = sum(w)
            for i in range(D):
                ref = sum(w[s] * v[s, g, i] for s in range(t + 1)) / tot
                assert o[t, h, i] == pytest.approx(ref, rel=1e-12, abs=1e-14)


def test_attention_special_cases():
    L, Hq, Hkv, D = 9, 16, 4, 8
    v = rng.normal(size=(L, Hkv, D))
    k = rng.normal(size=(L, Hkv, D))
    # L = 1: the only key is the query's own
    o1 = Lr.causal_attention(rng.normal(size=(1, Hq, D)), k[:1], v[:1])
    np.testing.assert_allclose(o1[0], np.repeat(v[0], 4, axis=0), rtol=1e-15)
    # q = 0: uniform weights, o_t = mean of v_0..t, for head h from kv head h // 4
    o0 = Lr.causal_attention(np.zeros((L, Hq, D)), k, v)
    means = np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None, None]
    np.testing.assert_allclose(o0, np.repeat(means, 4, axis=1), rtol=1e-13)


# ------------------------------------------------------------------------------------ rope
def test_rope_closed_form_and_passthrough():
    D = 256
    x = np.zeros((3, 1, D))
    x[:, 0, 0] = 1.0           # pair (0, 32): frequency 1
    x[:, 0, 31] = 1.0          # pair (31, 63): frequency 1e7^(-62/64)
    x[:, 0, 100] = 2.5         # beyond the rotary dims
    y = Lr.rope(x, np.array([0, 1, 5]))
    for i, p in enumerate((0, 1, 5)):
        assert y[i, 0, 0] == pytest.approx(math.cos(p), abs=1e-15)
        assert y[i, 0, 32] == pytest.approx(math.sin(p), abs=1e-15)
        f = 1e7 ** (-62 / 64)
        assert y[i, 0, 31] == pytest.approx(math.cos(p * f), abs=1e-15)
        assert y[i, 0, 63] == pytest.approx(math.sin(p * f), abs=1e-15)
        assert y[i, 0, 100] == 2.5


def test_rope_norm_and_relative_position():
    q = rng.normal(size=(1, 1, 256))
    k = rng.normal(size=(1, 1, 256))
    np.testing.assert_allclose(np.linalg.norm(Lr.rope(q, [17])), np.linalg.norm(q), rtol=1e-14)
    dots = []
    for p in (0, 10, 1000, 12345):
        dots.append(np.sum(Lr.rope(q, [p + 7]) * Lr.rope(k, [p])))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# ---------------------------------------------------------------------- z-gated norm, mixers
def test_zgated_norm_closed_form():
    L, H, d = 2, 3, 8
    o = np.ones((L, H, d)) * np.arange(1, H + 1)[None, :, None]      # constant per head
    w = rng.normal(1, 0.1, size=d)
    z = rng.normal(size=(L, H, d))
    y = Lr.zgated_norm(o, z, w, eps=0.0).reshape(L, H, d)
    np.testing.assert_allclose(y, w * z / (1 + np.exp(-z)), rtol=1e-14)


def test_lut_model_mixers_are_causal():
    # one GDN mixer and one attention mixer at full width with small L; synthetic weights
    import synth
    wg = synth.gdn_layer_weights(7, 0)
    wa = synth.attention_layer_weights(7, 3)
    x = synth.normal_f16(7, "x", 0, (8, 4096)).astype(np.float64)
    for mixer, w in ((model.gdn_mixer, wg), (model.attention_mixer, wa)):
        full = mixer(x, w)
        pre = mixer(x[:5], w)
        np.testing.assert_allclose(full[:5], pre, rtol=1e-10, atol=1e-12)
        x2 = x.copy()
        x2[6] += 1.0
        moved = mixer(x2, w)
        np.testing.assert_array_equal(moved[:6], full[:6])
        assert np.abs(moved[6:] - full[6:]).max() > 1e-3


def _const_lut6(n, k, value, seed):
    """A LUT-6 weight whose every entry is `value` (random indices into a constant table)."""
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 256, size=(n, k * 3 // 4), dtype=np.uint8)
    return packed, np.full((n // 16, 64), value, dtype=np.float16)


def test_swiglu_mlp_closed_form():
    """Constant weights gate = a, up = b, down = d give y_i = d * I * silu(a s) * b s with s the
    row sum of x: swapped gate/up operands or a missing SiLU factor would fail."""
    a, b, d, H, I = 0.25, -0.5, 0.125, 32, 48
    w = {"gate": _const_lut6(I, H, a, 1), "up": _const_lut6(I, H, b, 2),
         "down": _const_lut6(H, I, d, 3)}
    x = np.random.default_rng(4).standard_normal((5, H))
    s = x.sum(axis=1)
    expect = d * I * (a * s / (1 + np.exp(-a * s))) * (b * s)
    got = model.swiglu_mlp(x, w)
    assert np.allclose(got, np.repeat(expect[:, None], H, axis=1), rtol=1e-12, atol=0)


def test_decoder_layer_is_prenorm_residual():
    """A GDN layer whose mixer weights are zero is x + mlp(rmsnorm(x) * w_mlp): the residual
    carries x unchanged, and the MLP reads the normalised stream (the pre-norm block)."""
    import synth
    w = synth.gdn_layer_weights(5, 0)
    for name in ("qkv", "z", "out"):
        packed, lut = w[name]
        w[name] = (packed, np.zeros_like(lut))
    a, b, d = 2.0 ** -5, 2.0 ** -6, 2.0 ** -7          # exact in the fp16 tables
    w["gate"] = _const_lut6(12288, 4096, a, 6)
    w["up"] = _const_lut6(12288, 4096, b, 7)
    w["down"] = _const_lut6(4096, 12288, d, 8)
    x = synth.normal_f16(5, "x", 0, (3, 4096)).astype(np.float64)
    got = model.decoder_layer(x, w, attention=False)
    xn = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + 1e-6) * w["mlp_norm"].astype(np.float64)
    s = xn.sum(axis=1)
    mlp = d * 12288 * (a * s / (1 + np.exp(-a * s))) * (b * s)
    assert np.allclose(got, x + mlp[:, None], rtol=1e-10, atol=1e-12)


def test_attention_output_gate_closed_form():
    """Zero query/key weights make the causal softmax uniform (row t averages v over 0..t); with
    constant v = c_v, gate block (Q-proj rows 4096..8191) = c_g and O-proj = c_o, output row t is
    c_o * 4096 * c_v * mean_{p<=t} s_p * sigmoid(c_g * s_t), s the row sum of x.  Taking the gate
    from the first half of the Q-proj, or dropping the sigmoid, fails."""
    c_v, c_g, c_o = 2.0 ** -6, 2.0 ** -4, 2.0 ** -9                 # exact in the fp16 tables
    rng = np.random.default_rng(9)
    q_packed = rng.integers(0, 256, size=(8192, 3072), dtype=np.uint8)
    q_lut = np.zeros((512, 64), dtype=np.float16)
    q_lut[256:] = c_g                                                # gate heads only
    w = {"q": (q_packed, q_lut), "k": _const_lut6(1024, 4096, 0.0, 10),
         "v": _const_lut6(1024, 4096, c_v, 11), "o": _const_lut6(4096, 4096, c_o, 12)}
    x = rng.standard_normal((6, 4096)) * 0.05
    s = x.sum(axis=1)
    prefix_mean = np.cumsum(s) / np.arange(1, 7)
    expect = c_o * 4096 * c_v * prefix_mean / (1 + np.exp(-c_g * s))
    got = model.attention_mixer(x, w)
    assert np.allclose(got, np.repeat(expect[:, None], 4096, axis=1), rtol=1e-10, atol=0)


def test_gdn_mixer_closed_form():
    """The GDN mixer end to end on a case with a scalar closed form.  Constant QKV weights c1,
    conv passing only the current tap, zero a/b projections and A_log = dt_bias = 0 (so
    alpha = exp(-softplus(0)) = 1/2 and beta = sigmoid(0) = 1/2): every q, k, v row is constant,
    q = k = u_t 1 after the L2 norm with u_t = sigma_t / sqrt(128 sigma_t^2 + eps), sigma_t =
    SiLU(c1 s_t), and the state stays m_t 1 1^T with
        m_t = alpha m_{t-1} + beta u_t (sigma_t - 128 alpha u_t m_{t-1}),
    so o_t = sqrt(128) u_t m_t 1; the z-gated norm turns that into r_t w_o SiLU(c2 s_t) with
    r_t = o / sqrt(o^2 + eps) (o the constant entry), and the output projection c3 sums it."""
    import synth
    w = synth.gdn_layer_weights(11, 0)
    c1, c2, c3 = 2.0 ** -10, 2.0 ** -9, 2.0 ** -12
    w["qkv"] = _const_lut6(8192, 4096, c1, 21)
    w["z"] = _const_lut6(4096, 4096, c2, 22)
    w["out"] = _const_lut6(4096, 4096, c3, 23)
    w["a_w"] = np.zeros_like(w["a_w"])
    w["b_w"] = np.zeros_like(w["b_w"])
    w["A_log"] = np.zeros_like(w["A_log"])
    w["dt_bias"] = np.zeros_like(w["dt_bias"])
    conv = np.zeros_like(w["conv_w"])
    conv[:, 3] = 1.0                                          # the current position only
    w["conv_w"] = conv
    xn = np.random.default_rng(12).uniform(0.0, 1e-3, size=(6, 4096))
    s = xn.sum(axis=1)
    silu = lambda t: t / (1.0 + np.exp(-t))  # noqa: E731
    sigma = silu(c1 * s)
    u = sigma / np.sqrt(128 * sigma ** 2 + 1e-6)
    alpha = beta = 0.5
    m, expect = 0.0, []
    for t in range(6):
        m = alpha * m + beta * u[t] * (sigma[t] - 128 * alpha * u[t] * m)
        o = np.sqrt(128) * u[t] * m
        r = o / np.sqrt(o * o + 1e-6)
        y_sum = 32 * r * silu(c2 * s[t]) * float(np.sum(w["o_norm"].astype(np.float64)))
        expect.append(c3 * y_sum)
    got = model.gdn_mixer(xn, w)
    assert np.allclose(got, np.repeat(np.array(expect)[:, None], 4096, axis=1), rtol=1e-9, atol=0)

"""The C++ oracle against its numpy twin (CPU only).

Two independent writings of the same definitions (oracle/csrc in C++17, oracle/twin in numpy)
must agree: a dropped term, a wrong index or a transposed operand in either shows up here.
Floating-point results agree to fp64 rounding (1e-12 relative); integer work, the quantiser
(an exactly rounded algorithm) and the fp16 tables agree bit for bit.
"""
import numpy as np
import pytest

import synth
from oracle import layers as Lr
from oracle import lut6, model
from oracle import quantize as Q
from oracle.twin import layers as TLr
from oracle.twin import lut6 as Tlut6
from oracle.twin import model as Tmodel
from oracle.twin import quantize as TQ

rng = np.random.default_rng(77)
RTOL = 1e-12


def close(a, b, rtol=RTOL):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape
    scale = max(np.abs(b).max(), 1e-300)
    assert np.abs(a - b).max() <= rtol * scale, np.abs(a - b).max() / scale


def test_lut6_format():
    n, k = 48, 64
    idx = rng.integers(0, 64, size=(n, k), dtype=np.uint8)
    assert np.array_equal(lut6.pack(idx), Tlut6.pack(idx))
    packed = rng.integers(0, 256, size=(n, k * 3 // 4), dtype=np.uint8)
    assert np.array_equal(lut6.unpack(packed, k), Tlut6.unpack(packed, k))
    lut = rng.standard_normal((n // 16, 64)).astype(np.float16)
    assert np.array_equal(lut6.dequant(packed, lut, n, k), Tlut6.dequant(packed, lut, n, k))
    assert np.array_equal(lut6.dequant_f16(packed, lut, n, k).view(np.uint16),
                          Tlut6.dequant_f16(packed, lut, n, k).view(np.uint16))
    x = rng.standard_normal((37, k))
    close(lut6.linear(x, packed, lut, n), Tlut6.linear(x, packed, lut, n))
    assert lut6.storage_bits(4096, 4096) == Tlut6.storage_bits(4096, 4096)


def test_norms_and_elementwise():
    x = rng.standard_normal((9, 40)) * 3
    w = rng.standard_normal(40)
    close(Lr.rmsnorm(x, w), TLr.rmsnorm(x, w))
    close(Lr.l2norm(x), TLr.l2norm(x))
    for f, g in ((Lr.silu, TLr.silu), (Lr.sigmoid, TLr.sigmoid), (Lr.softplus, TLr.softplus)):
        close(f(x * 10), g(x * 10))


def test_conv_and_gates():
    x = rng.standard_normal((11, 24))
    w = rng.standard_normal((24, 4))
    close(Lr.causal_conv_silu(x, w), TLr.causal_conv_silu(x, w))
    close(Lr.causal_conv_silu(x[:2], w), TLr.causal_conv_silu(x[:2], w))
    a, b = rng.standard_normal((7, 5)) * 4, rng.standard_normal((7, 5)) * 4
    A_log, dt = rng.standard_normal(5), rng.standard_normal(5)
    for u, v in zip(Lr.gdn_gates(a, b, A_log, dt), TLr.gdn_gates(a, b, A_log, dt)):
        close(u, v)


@pytest.mark.parametrize("with_s0", [False, True])
def test_delta_rule(with_s0):
    L, Hk, Hv, dk, dv = 23, 2, 4, 8, 6
    q = TLr.l2norm(rng.standard_normal((L, Hk, dk)))
    k = TLr.l2norm(rng.standard_normal((L, Hk, dk)))
    v = rng.standard_normal((L, Hv, dv))
    alpha = rng.uniform(0.5, 1.0, (L, Hv))
    beta = rng.uniform(0.0, 1.0, (L, Hv))
    s0 = rng.standard_normal((Hv, dv, dk)) if with_s0 else None
    o, S = Lr.gated_delta_rule(q, k, v, alpha, beta, s0)
    to, tS = TLr.gated_delta_rule(q, k, v, alpha, beta, s0)
    close(o, to)
    close(S, tS)


def test_zgated_norm_and_rotary():
    o, z = rng.standard_normal((5, 3, 16)), rng.standard_normal((5, 3, 16))
    w = rng.standard_normal(16)
    close(Lr.zgated_norm(o, z, w), TLr.zgated_norm(o, z, w))
    x = rng.standard_normal((13, 3, 80))
    pos = rng.integers(0, 20000, size=13)
    close(Lr.rope(x, pos), TLr.rope(x, pos))
    for args in ((30, 0, 0, 0), (30, 4, 3, 5), (40, 0, 6, 2), (12, 11, 1, 1)):
        p3 = Lr.mrope_positions(*args)
        assert np.array_equal(p3, TLr.mrope_positions(*args))
        xx = rng.standard_normal((args[0], 2, 64))
        close(Lr.mrope(xx, p3), TLr.mrope(xx, p3))
    assert np.array_equal(Lr.mrope_planes(), TLr.mrope_planes())


def test_attention():
    L, Hq, Hkv, D = 45, 4, 2, 16
    q, k, v = (rng.standard_normal((L, h, D)) for h in (Hq, Hkv, Hkv))
    full = Lr.causal_attention(q, k, v)
    close(full, TLr.causal_attention(q, k, v))
    close(Lr.causal_attention(q, k, v, rows=(17, 40)), full[17:40])


def test_mlp_and_mixers_full_width():
    wg = synth.gdn_layer_weights(3, 0)
    wa = synth.attention_layer_weights(3, 3)
    x = synth.normal_f16(3, "twin.x", 0, (5, 4096)).astype(np.float64)
    close(model.swiglu_mlp(x, wg), Tmodel.swiglu_mlp(x, wg))
    close(model.gdn_mixer(x, wg), Tmodel.gdn_mixer(x, wg))
    close(model.attention_mixer(x, wa), Tmodel.attention_mixer(x, wa))
    p3 = Lr.mrope_positions(5, 1, 2, 2)
    close(model.attention_mixer(x, wa, p3), Tmodel.attention_mixer(x, wa, p3))
    close(model.decoder_layer(x, wg, False), Tmodel.decoder_layer(x, wg, False))


def test_prefill_four_layers():
    ids = synth.token_ids(5, 1, 6)[0]
    emb = synth.embedding_rows(0, ids)
    got = model.prefill(ids, emb, lambda l: synth.layer_weights(0, l), synth.final_norm_weight(0), n_layers=4)
    ref = Tmodel.prefill(ids, emb, lambda l: synth.layer_weights(0, l), synth.final_norm_weight(0), n_layers=4)
    close(got, ref, 1e-11)


def _fp16_group(kind, n=512):
    if kind == "normal":
        v = rng.standard_normal(n) * 0.02
    elif kind == "heavy":
        v = rng.standard_t(2, n) * 0.01
    elif kind == "levels":
        v = rng.choice([-0.5, -0.125, 0.0, 0.25, 1.0], size=n)
    elif kind == "tiny":       # subnormals, signed zeros and a few normals
        v = np.concatenate([rng.integers(-40, 40, n - 8) * 2.0 ** -24, [0.0, -0.0, -0.0, 0.0],
                            rng.standard_normal(4) * 1e-3])
    else:
        v = np.full(n, 0.375)
    return np.asarray(v, np.float16).astype(np.float64)


@pytest.mark.parametrize("kind", ["normal", "heavy", "levels", "tiny", "constant"])
def test_quantiser_bit_for_bit(kind):
    v = _fp16_group(kind)
    assert np.array_equal(Q.quantiles(v), TQ.quantiles(v))
    assert np.array_equal(Q.spread(v), TQ.spread(v))
    c = Q.initial_table(v)
    assert np.array_equal(c, TQ.initial_table(v))
    assert np.array_equal(Q.assign(v, c), TQ.assign(v, c))
    assert np.array_equal(Q.kmeans_round(v, c), TQ.kmeans_round(v, c))
    t, i = Q.quantize_group(v)
    tt, ti = TQ.quantize_group(v)
    assert np.array_equal(t.view(np.uint16), tt.view(np.uint16))
    assert np.array_equal(i, ti)


def test_quantize_matrix_bit_for_bit():
    w = (rng.standard_normal((32, 64)) * 0.02).astype(np.float16)
    p, l = Q.quantize(w)
    tp, tl = TQ.quantize(w)
    assert np.array_equal(p, tp)
    assert np.array_equal(l.view(np.uint16), tl.view(np.uint16))

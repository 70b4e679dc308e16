"""Pins of the oracle's prefill as a whole: how the layers compose (CPU only).

"Clef-Flash-ANE-LUT6", Model architecture: 32 layers, 24 Gated DeltaNet and 8 full-attention
layers with full attention every fourth layer; "clef-flash-LiteRT", Host contract: every
position's output of the final RMSNorm comes out.  Each test computes its expected value from a
closed form written here, not from the oracle.
"""
import numpy as np
import pytest

import synth
from oracle import model

EPS = 1e-6


def _rms(x, w):
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + EPS) * np.asarray(w, np.float64)


def _const_lut6(n, k, value, seed):
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 256, size=(n, k * 3 // 4), dtype=np.uint8)
    return packed, np.full((n // 16, 64), value, dtype=np.float16)


def _zero_table(w):
    packed, lut = w
    return packed, np.zeros_like(lut)


def _silenced(layer, seed=0):
    """Layer `layer`'s synthetic weights with its mixer output projection and MLP down
    projection at zero: the layer then passes its input through unchanged."""
    w = synth.layer_weights(seed, layer)
    w["out" if "out" in w else "o"] = _zero_table(w["out" if "out" in w else "o"])
    w["down"] = _zero_table(w["down"])
    return w


def _ids_rows(L, seed=3):
    ids = synth.token_ids(seed, 1, L)[0]
    return ids, synth.embedding_rows(0, ids).astype(np.float64)


def test_layer_phase_every_fourth_layer():
    """Full attention every fourth layer: layers 3, 7, ..., 31 (three Gated DeltaNet layers, then
    one attention layer), 8 of 32; layer 0 is a Gated DeltaNet layer."""
    kinds = [model.is_attention_layer(l) for l in range(32)]
    assert sum(kinds) == 8 and kinds.count(False) == 24
    assert [l for l in range(32) if kinds[l]] == list(range(3, 32, 4))
    assert not kinds[0] and kinds[3]


def test_prefill_with_silent_layers_is_the_final_norm_of_the_embeddings():
    """With every mixer and MLP output at zero the residual stream carries the embedding rows
    through all layers, and the prefill returns their final RMSNorm."""
    ids, emb = _ids_rows(5)
    fn = synth.final_norm_weight(0)
    got = model.prefill(ids, emb, _silenced, fn, n_layers=4)
    np.testing.assert_allclose(got, _rms(emb, fn.astype(np.float64)), rtol=1e-12, atol=0)


def test_prefill_applies_the_layers_in_order():
    """Zero mixers and constant SwiGLU weights (a_l, b_l, d_l) per layer: layer l maps each row h
    to h + d_l I silu(a_l s) b_l s, s the row sum of rmsnorm(h) * w_mlp.  The map is not linear,
    so the four layers give a different result in any other order; the reversed order is checked
    to differ, so the test can tell."""
    # d_l small enough that each layer's addition is comparable to the embedding rows, so every
    # layer moves the row sums the next one sees (all constants exact in fp16)
    consts = [(2.0 ** -5, 2.0 ** -6, 2.0 ** -20), (2.0 ** -4, -(2.0 ** -6), 2.0 ** -21),
              (-(2.0 ** -5), 2.0 ** -5, 2.0 ** -19), (2.0 ** -3, 2.0 ** -7, -(2.0 ** -20))]

    def weights(l):
        w = synth.layer_weights(0, l)
        w["out" if "out" in w else "o"] = _zero_table(w["out" if "out" in w else "o"])
        a, b, d = consts[l]
        w["gate"] = _const_lut6(12288, 4096, a, 10 + l)
        w["up"] = _const_lut6(12288, 4096, b, 20 + l)
        w["down"] = _const_lut6(4096, 12288, d, 30 + l)
        return w

    ids, emb = _ids_rows(3)
    fn = synth.final_norm_weight(0)
    got = model.prefill(ids, emb, weights, fn, n_layers=4)

    def closed_form(order):
        h = emb.copy()
        for l in order:
            a, b, d = consts[l]
            s = _rms(h, synth.layer_weights(0, l)["mlp_norm"]).sum(axis=1)
            h = h + (d * 12288 * (a * s / (1 + np.exp(-a * s))) * (b * s))[:, None]
        return _rms(h, fn.astype(np.float64))

    expect = closed_form([0, 1, 2, 3])
    np.testing.assert_allclose(got, expect, rtol=1e-9, atol=1e-12)
    assert np.abs(closed_form([3, 2, 1, 0]) - expect).max() > 0.1 * np.abs(expect).max()


def test_prefill_runs_attention_at_layer_three():
    """Layers 0-2 silent, layer 3 an attention layer with zero query/key weights, constant v
    (c_v), gate block (c_g) and O-projection (c_o), and a silent MLP: the output is the final
    norm of x + c_o 4096 c_v mean_{p<=t} s_p sigmoid(c_g s_t), s the row sums of
    rmsnorm(x) * w_attn_norm.  A prefill that put the attention layer elsewhere in the group of
    four would not find its weights where it needs them, or would give another result."""
    c_v, c_g, c_o = 2.0 ** -6, 2.0 ** -4, 2.0 ** -9
    rng = np.random.default_rng(9)

    def weights(l):
        if l != 3:
            return _silenced(l)
        w = synth.layer_weights(0, 3)
        q_packed = rng.integers(0, 256, size=(8192, 3072), dtype=np.uint8)
        q_lut = np.zeros((512, 64), dtype=np.float16)
        q_lut[256:] = c_g
        w.update(q=(q_packed, q_lut), k=_const_lut6(1024, 4096, 0.0, 10),
                 v=_const_lut6(1024, 4096, c_v, 11), o=_const_lut6(4096, 4096, c_o, 12))
        w["down"] = _zero_table(w["down"])
        return w

    ids, emb = _ids_rows(6)
    fn = synth.final_norm_weight(0)
    got = model.prefill(ids, emb, weights, fn, n_layers=4)
    s = _rms(emb, synth.layer_weights(0, 3)["attn_norm"]).sum(axis=1)
    prefix_mean = np.cumsum(s) / np.arange(1, 7)
    mix = c_o * 4096 * c_v * prefix_mean / (1 + np.exp(-c_g * s))
    expect = _rms(emb + mix[:, None], fn.astype(np.float64))
    np.testing.assert_allclose(got, expect, rtol=1e-9, atol=1e-12)
    # the mixer is visible in the result (the test has power)
    assert np.abs(expect - _rms(emb, fn.astype(np.float64))).max() > 1e-3


def test_prefill_refuses_weights_of_the_wrong_kind():
    ids, emb = _ids_rows(4)
    with pytest.raises(ValueError):
        # attention weights where the phase puts a Gated DeltaNet layer
        model.prefill(ids, emb, lambda l: synth.layer_weights(0, 3), synth.final_norm_weight(0),
                      n_layers=1)

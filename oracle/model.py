"""Oracle decoder layers and the 32-layer hybrid prefill: thin marshalling over the C++ oracle
(oracle/csrc/model.cpp, fp64).

Weights come as a dict per layer (the names of synth's recipe): LUT-6 linears as
(packed [n, k*3/4] uint8, lut [n/16, 64] fp16) pairs, the rest as fp16 arrays.  This module only
lays them out as the C structs and passes pointers.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import Layer, Lut6Weight, check, contig, f16_bits, f64, lib, ptr

GDN_HK, GDN_HV, GDN_D = 16, 32, 128
ATT_HQ, ATT_HKV, ATT_D = 16, 4, 256

_LUT6_NAMES = ("qkv", "z", "out", "q", "k", "v", "o", "gate", "up", "down")
_F16_NAMES = ("attn_norm", "mlp_norm", "a_w", "b_w", "A_log", "dt_bias", "conv_w", "o_norm")


def _layer_struct(w, attention, keep):
    """The orc_layer struct of a weight dict; `keep` holds the arrays the pointers point into."""
    s = Layer()
    s.attention = 1 if attention else 0
    for name in _LUT6_NAMES:
        if name in w:
            packed, lut = w[name]
            p, t = contig(packed, np.uint8), f16_bits(lut)
            keep += [p, t]
            setattr(s, name, Lut6Weight(p.ctypes.data, t.ctypes.data, t.shape[0] * 16, p.shape[1] * 4 // 3))
    for name in _F16_NAMES:
        if name in w:
            a = f16_bits(w[name])
            keep.append(a)
            setattr(s, name, a.ctypes.data)
    return s


def _positions(L, positions, keep):
    if positions is None:
        return None, None
    pos = np.asarray(positions)
    if pos.ndim == 2:
        p3 = contig(pos, np.int64).reshape(L, 3)
        keep.append(p3)
        return None, p3
    p = f64(pos).reshape(L)
    keep.append(p)
    return p, None


def swiglu_mlp(xn, w):
    """SwiGLU MLP: down(SiLU(x W_gate^T) * (x W_up^T)); all three LUT-6."""
    x = f64(xn)
    L, H = x.shape
    keep = []
    s = _layer_struct(w, False, keep)
    out = np.empty((L, H))
    check(lib().orc_swiglu_mlp(ptr(x), L, H, ctypes.byref(s), ptr(out)), "swiglu_mlp")
    return out


def gdn_mixer(xn, w):
    """Gated DeltaNet mixer on one request.  xn: normalised input [L, 4096] -> [L, 4096]."""
    x = f64(xn)
    L, H = x.shape
    keep = []
    s = _layer_struct(w, False, keep)
    out = np.empty((L, H))
    check(lib().orc_gdn_mixer(ptr(x), L, H, ctypes.byref(s), ptr(out)), "gdn_mixer")
    return out


def attention_mixer(xn, w, positions=None):
    """Gated full-attention mixer on one request.  xn: [L, 4096]; positions [L] or [L, 3]."""
    x = f64(xn)
    L, H = x.shape
    keep = []
    s = _layer_struct(w, True, keep)
    pos, pos3 = _positions(L, positions, keep)
    out = np.empty((L, H))
    check(lib().orc_attention_mixer(ptr(x), L, H, ctypes.byref(s), ptr(pos), ptr(pos3), ptr(out)),
          "attention_mixer")
    return out


def decoder_layer(x, w, attention: bool, positions=None):
    """One pre-norm residual decoder layer on one request: x [L, 4096] -> [L, 4096]."""
    xx = f64(x)
    L, H = xx.shape
    keep = []
    s = _layer_struct(w, attention, keep)
    pos, pos3 = _positions(L, positions, keep)
    out = np.empty((L, H))
    check(lib().orc_decoder_layer(ptr(xx), L, H, ctypes.byref(s), ptr(pos), ptr(pos3), ptr(out)),
          "decoder_layer")
    return out


def is_attention_layer(layer: int) -> bool:
    return bool(lib().orc_is_attention_layer(layer))


def prefill(ids, embed_rows, layer_weights, final_norm, n_layers=32, positions=None):
    """The hybrid prefill of one request: ids [L] -> final-norm hidden [L, 4096] (float64).

    `embed_rows` is [L, 4096] (the table's rows at `ids`, gathered by the caller; a request with a
    picture passes the picture's rows where its image tokens sit); `layer_weights(l)` returns
    layer l's weight dict; `positions` are M-RoPE positions [L, 3] (or [L], or None: 0 .. L-1).
    """
    x = f64(embed_rows)
    L, H = x.shape
    assert L == len(ids)
    keep = []
    structs = (Layer * n_layers)()
    for layer in range(n_layers):
        structs[layer] = _layer_struct(layer_weights(layer), is_attention_layer(layer), keep)
    fn = f16_bits(final_norm)
    pos, pos3 = _positions(L, positions, keep)
    out = np.empty((L, H))
    check(lib().orc_prefill(ptr(x), L, H, structs, n_layers, ptr(fn), ptr(pos), ptr(pos3), ptr(out)),
          "prefill")
    return out

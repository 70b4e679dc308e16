"""Decoder layers and the 32-layer prefill: the numpy twin of the C++ oracle (float64).

Architecture ("Clef-Flash-ANE-LUT6" §Model architecture; "clef-flash-LiteRT" §Provenance):
32 layers of hidden size 4,096 and MLP size 12,288; 24 Gated DeltaNet layers and 8 gated
full-attention layers, full attention every fourth layer (layers 3, 7, ..., 31).  Every large
linear is LUT-6 (§Weight precision).  Each layer is a pre-norm residual block (adopted reading;
the pages are silent on it):  h = x + mixer(rmsnorm(x)),  y = h + mlp(rmsnorm(h)).

Weights come as a dict per layer: LUT-6 linears as (packed [n, k*3/4] uint8, lut [n/16, 64] fp16)
pairs, the rest as fp16 arrays.  End-to-end activations are parity unpinned against the pages
(no page prints one); the layers' parts are pinned piecewise by the oracle's own tests.
"""
from __future__ import annotations

import numpy as np

from . import layers as Lr
from . import lut6

GDN_HK, GDN_HV, GDN_D = 16, 32, 128
ATT_HQ, ATT_HKV, ATT_D = 16, 4, 256


def _lin(x, wt):
    packed, lut = wt
    n = lut.shape[0] * lut6.GROUP_ROWS
    return lut6.linear(x, packed, lut, n)


def swiglu_mlp(xn, w):
    """SwiGLU MLP: down(SiLU(x W_gate^T) * (x W_up^T)); all three LUT-6 ("Clef-Flash-ANE-LUT6"
    §Weight precision lists MLP gate/up/down among the LUT-6 layers)."""
    return _lin(Lr.silu(_lin(xn, w["gate"])) * _lin(xn, w["up"]), w["down"])


def gdn_mixer(xn, w, return_parts=False):
    """Gated DeltaNet mixer on one request.  xn: normalised input [L, 4096].

    QKV (4096 -> 8192 = q 2048 | k 2048 | v 4096) and Z (4096 -> 4096) are LUT-6; the gate
    projections a, b (4096 -> 32 each) are FP16 ("Clef-Flash-ANE-LUT6" §Weight precision).
    Conv + SiLU on all 8,192 QKV channels, per-head L2 norm of q and k, gates, the delta rule,
    the z-gated RMSNorm, then the LUT-6 output projection (4096 -> 4096).
    """
    xn = Lr.f64(xn)
    L = xn.shape[0]
    qkv = _lin(xn, w["qkv"])
    z = _lin(xn, w["z"])
    a = xn @ Lr.f64(w["a_w"]).T
    b = xn @ Lr.f64(w["b_w"]).T
    c = Lr.causal_conv_silu(qkv, w["conv_w"])
    qk = GDN_HK * GDN_D
    q = Lr.l2norm(c[:, :qk].reshape(L, GDN_HK, GDN_D))
    k = Lr.l2norm(c[:, qk:2 * qk].reshape(L, GDN_HK, GDN_D))
    v = c[:, 2 * qk:].reshape(L, GDN_HV, GDN_D)
    alpha, beta = Lr.gdn_gates(a, b, w["A_log"], w["dt_bias"])
    o, S = Lr.gated_delta_rule(q, k, v, alpha, beta)
    y = Lr.zgated_norm(o, z.reshape(L, GDN_HV, GDN_D), w["o_norm"])
    out = _lin(y, w["out"])
    if return_parts:
        return out, dict(qkv=qkv, z=z, a=a, b=b, q=q, k=k, v=v, alpha=alpha, beta=beta, o=o,
                         S=S, y=y)
    return out


def attention_mixer(xn, w, positions=None, return_parts=False):
    """Gated full-attention mixer on one request.  xn: [L, 4096].

    Q-proj 4096 -> 8192 holds the 16 query heads (columns 0..4095) and 16 output-gate heads
    (4096..8191): adopted reading of "gated full-attention layers" ("clef-flash-LiteRT"
    §Provenance), the only one that makes the model's stored LUT-6 size match the 4.86 GiB the
    "Clef-Flash-ANE-LUT6" card gives for its text programs.  K, V 4096 -> 1024 (4 heads x 256),
    rotary on the first 64 dims of q and k, causal GQA softmax, o * sigmoid(gate), O-proj.
    """
    xn = Lr.f64(xn)
    L = xn.shape[0]
    pos = np.arange(L) if positions is None else np.asarray(positions)
    rot = Lr.mrope if pos.ndim == 2 else Lr.rope       # [L, 3] M-RoPE planes or [L] positions
    qg = _lin(xn, w["q"])
    q = qg[:, :ATT_HQ * ATT_D].reshape(L, ATT_HQ, ATT_D)
    gate = qg[:, ATT_HQ * ATT_D:]
    k = _lin(xn, w["k"]).reshape(L, ATT_HKV, ATT_D)
    v = _lin(xn, w["v"]).reshape(L, ATT_HKV, ATT_D)
    qr = rot(q, pos)
    kr = rot(k, pos)
    o = Lr.causal_attention(qr, kr, v).reshape(L, ATT_HQ * ATT_D)
    og = o * Lr.sigmoid(gate)
    out = _lin(og, w["o"])
    if return_parts:
        return out, dict(qg=qg, q=q, k=k, v=v, o=o, og=og)
    return out


def decoder_layer(x, w, attention: bool, positions=None):
    """One pre-norm residual decoder layer on one request: x [L, 4096] -> [L, 4096].
    `positions`: rotary positions of the attention layers ([L], or [L, 3] M-RoPE planes;
    default 0 .. L - 1)."""
    x = Lr.f64(x)
    xn = Lr.rmsnorm(x, w["attn_norm"])
    h = x + (attention_mixer(xn, w, positions) if attention else gdn_mixer(xn, w))
    return h + swiglu_mlp(Lr.rmsnorm(h, w["mlp_norm"]), w)


def is_attention_layer(layer: int) -> bool:
    return layer % 4 == 3


def prefill(ids, embed_rows, layer_weights, final_norm, n_layers=32, positions=None):
    """The hybrid prefill of one request: ids [L] -> final-norm hidden [L, 4096] (float64).

    "clef-flash-LiteRT" §Host contract steps 4-6: embedding rows at the request's ids in, every
    position's output of the final RMSNorm out, each call from an empty state.  `embed_rows` is [L, 4096] (the table's rows at `ids`, gathered by the caller);
    `layer_weights(l)` returns layer l's weight dict.  A request with a picture passes the
    picture's rows in place of the table's rows where its <|image_pad|> tokens sit (step 4) and its
    M-RoPE positions ([L, 3], :func:`oracle.layers.mrope_positions`; step 5).
    """
    x = Lr.f64(embed_rows)
    assert x.shape[0] == len(ids)
    for layer in range(n_layers):
        x = decoder_layer(x, layer_weights(layer), is_attention_layer(layer), positions)
    return Lr.rmsnorm(x, final_norm)

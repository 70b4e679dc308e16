"""Seeded synthetic inputs for the clef-flash prefill (shared by the oracle side and the CUDA side).

Holds no arithmetic of the prefill method: it only draws numbers.  The drawing is done by
``synth.c`` (splitmix64 counter stream, Box-Muller normals, Lemire bounded integers); this module
loads it with ctypes and lays the draws out as numpy arrays with the model's shapes.

Recipe of every tensor (name, distribution, shape) is in :func:`layer_recipe` and
:func:`model_inputs`; the model shapes are those of the clef-flash text backbone (hidden 4,096,
MLP 12,288, 32 layers, vocabulary 248,320) from the clef-flash-ane-lut6 model card
(§Model architecture).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None

HIDDEN = 4096
INTER = 12288
N_LAYERS = 32
VOCAB = 248320
GDN_QK = 2048      # 16 key heads x 128
GDN_V = 4096       # 32 value heads x 128
GDN_HV = 32
ATT_Q = 4096       # 16 query heads x 256
ATT_KV = 1024      # 4 kv heads x 256


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, src, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u64, i64, cp, d = ctypes.c_uint64, ctypes.c_int64, ctypes.c_char_p, ctypes.c_double
        vp = ctypes.c_void_p
        for fn in ("synth_normal_f16", "synth_normal_f32", "synth_normal_f64"):
            getattr(lib, fn).argtypes = [u64, cp, i64, d, d, vp, i64]
            getattr(lib, fn).restype = None
        lib.synth_bytes.argtypes = [u64, cp, i64, vp, i64]
        lib.synth_uniform_int.argtypes = [u64, cp, i64, ctypes.c_uint32, vp, i64]
        lib.synth_codes6.argtypes = [u64, cp, i64, vp, i64]
        lib.synth_normal_f16_range.argtypes = [u64, cp, i64, d, d, vp, i64, i64]
        lib.synth_normal_f16_range.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def normal_f16(seed, name, layer, shape, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float16)
    _load().synth_normal_f16(seed, name.encode(), layer, float(mean), float(std), _ptr(out), out.size)
    return out


def normal_f32(seed, name, layer, shape, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(seed, name.encode(), layer, float(mean), float(std), _ptr(out), out.size)
    return out


def normal_f64(seed, name, layer, shape, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float64)
    _load().synth_normal_f64(seed, name.encode(), layer, float(mean), float(std), _ptr(out), out.size)
    return out


def random_bytes(seed, name, layer, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint8)
    _load().synth_bytes(seed, name.encode(), layer, _ptr(out), out.size)
    return out


def uniform_int(seed, name, layer, shape, bound) -> np.ndarray:
    out = np.empty(shape, dtype=np.int32)
    _load().synth_uniform_int(seed, name.encode(), layer, int(bound), _ptr(out), out.size)
    return out


def codes6(seed, name, layer, shape) -> np.ndarray:
    """Uniform 6-bit codes (0..63), one byte each: the top 6 bits of each draw."""
    out = np.empty(shape, dtype=np.uint8)
    _load().synth_codes6(seed, name.encode(), layer, _ptr(out), out.size)
    return out


# ----------------------------------------------------------------------------------------------
# LUT-6 weights.  Packed stream [n, k*3/4] bytes; tables [n/16, 64] fp16 N(0, 0.02).
# Uniform random bytes are uniform 6-bit codes under any bijective 4-in-3 packing, so the packed
# stream is drawn directly as bytes (the codes are whatever unpacking the bytes yields).
# ----------------------------------------------------------------------------------------------
def lut6_weight(seed, name, layer, n, k, table_std=0.02):
    assert n % 16 == 0 and k % 4 == 0
    packed = random_bytes(seed, name + ".packed", layer, (n, k * 3 // 4))
    lut = normal_f16(seed, name + ".lut", layer, (n // 16, 64), 0.0, table_std)
    return packed, lut


def norm_weight(seed, name, layer, n):
    """RMSNorm weights 1 + N(0, 0.02), fp16."""
    return normal_f16(seed, name, layer, (n,), 1.0, 0.02)


def is_attention_layer(layer: int) -> bool:
    """Full attention every fourth layer (layers 3, 7, ..., 31); the rest are Gated DeltaNet."""
    return layer % 4 == 3


def gdn_layer_weights(seed, layer, hidden=HIDDEN, inter=INTER):
    """All parameters of one Gated DeltaNet decoder layer (names are the recipe)."""
    w = {}
    w["attn_norm"] = norm_weight(seed, "attn_norm", layer, hidden)
    w["qkv"] = lut6_weight(seed, "gdn.qkv", layer, 2 * GDN_QK + GDN_V, hidden)
    w["z"] = lut6_weight(seed, "gdn.z", layer, GDN_V, hidden)
    w["a_w"] = normal_f16(seed, "gdn.a_w", layer, (GDN_HV, hidden), 0.0, hidden ** -0.5)
    w["b_w"] = normal_f16(seed, "gdn.b_w", layer, (GDN_HV, hidden), 0.0, hidden ** -0.5)
    # decay parameters: A_log around ln 0.1 and dt_bias around 0 (per value head, fp16)
    w["A_log"] = normal_f16(seed, "gdn.A_log", layer, (GDN_HV,), float(np.log(0.1)), 0.1)
    w["dt_bias"] = normal_f16(seed, "gdn.dt_bias", layer, (GDN_HV,), 0.0, 0.1)
    w["conv_w"] = normal_f16(seed, "gdn.conv_w", layer, (2 * GDN_QK + GDN_V, 4), 0.0, 0.5)
    w["o_norm"] = norm_weight(seed, "gdn.o_norm", layer, 128)
    w["out"] = lut6_weight(seed, "gdn.out", layer, hidden, GDN_V)
    w.update(mlp_weights(seed, layer, hidden, inter))
    return w


def attention_layer_weights(seed, layer, hidden=HIDDEN, inter=INTER):
    """All parameters of one gated full-attention decoder layer."""
    w = {}
    w["attn_norm"] = norm_weight(seed, "attn_norm", layer, hidden)
    w["q"] = lut6_weight(seed, "att.q", layer, 2 * ATT_Q, hidden)   # query heads || gate heads
    w["k"] = lut6_weight(seed, "att.k", layer, ATT_KV, hidden)
    w["v"] = lut6_weight(seed, "att.v", layer, ATT_KV, hidden)
    w["o"] = lut6_weight(seed, "att.o", layer, hidden, ATT_Q)
    w.update(mlp_weights(seed, layer, hidden, inter))
    return w


def mlp_weights(seed, layer, hidden=HIDDEN, inter=INTER):
    return {
        "mlp_norm": norm_weight(seed, "mlp_norm", layer, hidden),
        "gate": lut6_weight(seed, "mlp.gate", layer, inter, hidden),
        "up": lut6_weight(seed, "mlp.up", layer, inter, hidden),
        "down": lut6_weight(seed, "mlp.down", layer, hidden, inter),
    }


def layer_weights(seed, layer):
    return attention_layer_weights(seed, layer) if is_attention_layer(layer) else gdn_layer_weights(seed, layer)


def final_norm_weight(seed):
    return norm_weight(seed, "final_norm", -1, HIDDEN)


def embedding_table(seed):
    """Token embeddings [248320, 4096] fp16, N(0, 0.02) (2.03 GB)."""
    return normal_f16(seed, "embed", -1, (VOCAB, HIDDEN), 0.0, 0.02)


def embedding_rows(seed, ids):
    """Only the rows of the embedding table at `ids` (the same values as embedding_table)."""
    ids = np.asarray(ids).reshape(-1)
    lib = _load()
    out = np.empty((ids.size, HIDDEN), dtype=np.float16)
    for r, t in enumerate(ids):
        lib.synth_normal_f16_range(seed, b"embed", -1, 0.0, 0.02, _ptr(out[r]), int(t) * HIDDEN, HIDDEN)
    return out


def token_ids(seed, batch, length, name="ids"):
    """Uniform token ids over the 248,320-token vocabulary, int32 [batch, length]."""
    return uniform_int(seed, name, -1, (batch, length), VOCAB)


# ----------------------------------------------------------------------------------------------
# Joint schema head (synthetic weights; width 1,024, 16 heads, 4 decoder + 2 routing layers).
# Projections N(0, 1/fan_in), norm weights 1 + N(0, 0.02), embeddings N(0, 0.5), all fp16.
# ----------------------------------------------------------------------------------------------
HEAD_D = 1024
HEAD_FF = 4096


def head_layer_weights(seed, name, layer):
    d, ff = HEAD_D, HEAD_FF
    w = {"norm1": norm_weight(seed, f"{name}.norm1", layer, d),
         "norm2": norm_weight(seed, f"{name}.norm2", layer, d)}
    for p in ("wq", "wk", "wv", "wo"):
        w[p] = normal_f16(seed, f"{name}.{p}", layer, (d, d), 0.0, d ** -0.5)
    w["wg"] = normal_f16(seed, f"{name}.wg", layer, (ff, d), 0.0, d ** -0.5)
    w["wu"] = normal_f16(seed, f"{name}.wu", layer, (ff, d), 0.0, d ** -0.5)
    w["wd"] = normal_f16(seed, f"{name}.wd", layer, (d, ff), 0.0, ff ** -0.5)
    return w


def head_weights(seed):
    """All parameters of the joint schema head (names are the recipe)."""
    d = HEAD_D
    w = {"w_mem": normal_f16(seed, "head.w_mem", -1, (d, HIDDEN), 0.0, HIDDEN ** -0.5),
         "w_in": normal_f16(seed, "head.w_in", -1, (d, HIDDEN), 0.0, HIDDEN ** -0.5),
         "w_lex": normal_f16(seed, "head.w_lex", -1, (d, HIDDEN), 0.0, HIDDEN ** -0.5),
         "e_qtype": normal_f16(seed, "head.e_qtype", -1, (3, d), 0.0, 0.5),
         "e_opt": normal_f16(seed, "head.e_opt", -1, (d,), 0.0, 0.5),
         "e_glob": normal_f16(seed, "head.e_glob", -1, (d,), 0.0, 0.5),
         "norm_f": norm_weight(seed, "head.norm_f", -1, d),
         "w_opt": normal_f16(seed, "head.w_opt", -1, (d, d), 0.0, d ** -0.5),
         "w_qst": normal_f16(seed, "head.w_qst", -1, (d, d), 0.0, d ** -0.5)}
    w["dec"] = [head_layer_weights(seed, "head.dec", l) for l in range(4)]
    w["route"] = [head_layer_weights(seed, "head.route", l) for l in range(2)]
    return w


def head_request(seed, T, questions):
    """A synthetic decision request's head inputs for T hidden rows: `questions` is a list of
    option counts.  Spans are drawn as disjoint runs of positions (questions' spans, then each
    option's), the global row is the last position; lexical rows N(0, 0.02) (the size of an
    lm_head row mean).  Returns a dict of numpy arrays (q_avg, o_avg, g_avg, lexical, member,
    type_ids, q_valid, o_valid, key_valid, q_span, o_span)."""
    Q, O = len(questions), int(sum(questions))
    lens = uniform_int(seed, "head.span_len", -1, (Q + O,), 7) + 2      # spans of 2..8 positions
    starts = uniform_int(seed, "head.span_gap", -1, (Q + O,), 3)
    q_avg = np.zeros((Q, T))
    o_avg = np.zeros((O, T))
    pos, spans = 1, []
    for i in range(Q + O):
        pos += int(starts[i])
        spans.append((pos, pos + int(lens[i])))
        pos += int(lens[i])
    assert pos < T, "T too short for the spans"
    for q in range(Q):
        a, b = spans[q]
        q_avg[q, a:b] = 1.0 / (b - a)
    member = np.zeros((Q, O), dtype=np.uint8)
    o = 0
    for q, n in enumerate(questions):
        for _ in range(n):
            a, b = spans[Q + o]
            o_avg[o, a:b] = 1.0 / (b - a)
            member[q, o] = 1
            o += 1
    g_avg = np.zeros(T)
    g_avg[T - 1] = 1.0
    return {"q_avg": q_avg, "o_avg": o_avg, "g_avg": g_avg,
            "lexical": normal_f64(seed, "head.lexical", -1, (O, HIDDEN), 0.0, 0.02),
            "member": member, "type_ids": (uniform_int(seed, "head.type", -1, (Q,), 3)),
            "q_valid": np.ones(Q, dtype=np.uint8), "o_valid": np.ones(O, dtype=np.uint8),
            "key_valid": np.ones(T, dtype=np.uint8),
            "q_span": spans[:Q], "o_span": spans[Q:]}

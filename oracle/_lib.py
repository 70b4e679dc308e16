"""ctypes loader of the C++ oracle (liboracle.so) and array marshalling.  Test infrastructure only.

Nothing here computes: it builds the library if needed, declares the signatures of
oracle/csrc/oracle.h, and passes numpy arrays as plain pointers.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

_lib = None

c_i64, c_i32, c_d = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
vp = ctypes.c_void_p


class Lut6Weight(ctypes.Structure):
    _fields_ = [("packed", vp), ("lut", vp), ("n", c_i64), ("k", c_i64)]


class Layer(ctypes.Structure):
    _fields_ = [
        ("attention", c_i32),
        ("attn_norm", vp), ("mlp_norm", vp),
        ("qkv", Lut6Weight), ("z", Lut6Weight), ("out", Lut6Weight),
        ("a_w", vp), ("b_w", vp), ("A_log", vp), ("dt_bias", vp), ("conv_w", vp), ("o_norm", vp),
        ("q", Lut6Weight), ("k", Lut6Weight), ("v", Lut6Weight), ("o", Lut6Weight),
        ("gate", Lut6Weight), ("up", Lut6Weight), ("down", Lut6Weight),
    ]


_SIGS = {
    "orc_last_error": (ctypes.c_char_p, []),
    "orc_num_threads": (c_i32, []),
    "orc_lut6_pack": (ctypes.c_int, [vp, c_i64, c_i64, vp]),
    "orc_lut6_unpack": (ctypes.c_int, [vp, c_i64, c_i64, vp]),
    "orc_lut6_dequant": (ctypes.c_int, [vp, vp, c_i64, c_i64, vp]),
    "orc_lut6_dequant_f16": (ctypes.c_int, [vp, vp, c_i64, c_i64, vp]),
    "orc_lut6_linear": (ctypes.c_int, [vp, c_i64, c_i64, vp, vp, c_i64, vp]),
    "orc_lut6_storage_bits": (c_i64, [c_i64, c_i64]),
    "orc_silu": (None, [vp, c_i64, vp]),
    "orc_sigmoid": (None, [vp, c_i64, vp]),
    "orc_softplus": (None, [vp, c_i64, vp]),
    "orc_rmsnorm": (None, [vp, c_i64, c_i64, vp, c_d, vp]),
    "orc_l2norm": (None, [vp, c_i64, c_i64, c_d, vp]),
    "orc_conv_silu": (None, [vp, c_i64, c_i64, vp, c_i64, vp]),
    "orc_gdn_gates": (None, [vp, vp, c_i64, c_i64, vp, vp, vp, vp]),
    "orc_gated_delta_rule": (ctypes.c_int, [vp] * 6 + [c_i64] * 5 + [vp, vp]),
    "orc_zgated_norm": (None, [vp, vp, c_i64, c_i64, c_i64, vp, c_d, vp]),
    "orc_rope": (None, [vp, c_i64, c_i64, c_i64, vp, c_i64, c_d, vp]),
    "orc_mrope_planes": (None, [c_i64, vp]),
    "orc_mrope_positions": (ctypes.c_int, [c_i64] * 4 + [vp]),
    "orc_mrope": (None, [vp, c_i64, c_i64, c_i64, vp, c_i64, c_d, vp]),
    "orc_causal_attention": (ctypes.c_int, [vp, vp, vp] + [c_i64] * 6 + [vp]),
    "orc_swiglu_mlp": (ctypes.c_int, [vp, c_i64, c_i64, ctypes.POINTER(Layer), vp]),
    "orc_gdn_mixer": (ctypes.c_int, [vp, c_i64, c_i64, ctypes.POINTER(Layer), vp]),
    "orc_attention_mixer": (ctypes.c_int, [vp, c_i64, c_i64, ctypes.POINTER(Layer), vp, vp, vp]),
    "orc_decoder_layer": (ctypes.c_int, [vp, c_i64, c_i64, ctypes.POINTER(Layer), vp, vp, vp]),
    "orc_is_attention_layer": (c_i32, [c_i64]),
    "orc_prefill": (ctypes.c_int, [vp, c_i64, c_i64, ctypes.POINTER(Layer), c_i64, vp, vp, vp, vp]),
    "orc_quant_quantiles": (None, [vp, c_i64, vp]),
    "orc_quant_spread": (None, [vp, c_i64, vp]),
    "orc_quant_initial_table": (None, [vp, c_i64, vp]),
    "orc_quant_assign": (None, [vp, c_i64, vp, c_i64, vp]),
    "orc_quant_kmeans_round": (None, [vp, c_i64, vp, c_i64]),
    "orc_quant_group": (None, [vp, c_i64, c_i32, vp, vp]),
    "orc_lut6_quantize": (ctypes.c_int, [vp, c_i64, c_i64, c_i32, vp, vp]),
    "orc_joint_head": (ctypes.c_int, [vp, vp, c_i64, vp, vp, vp, vp, vp, vp, vp, vp, c_i64, c_i64, vp,
                                      vp, vp]),
}


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(rc: int, where: str) -> None:
    if rc != 0:
        raise ValueError(f"{where}: {lib().orc_last_error().decode()}")


def f64(a) -> np.ndarray:
    """A C-contiguous float64 copy or view of `a` (fp16 values widen exactly)."""
    return np.ascontiguousarray(a, dtype=np.float64)


def contig(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def f16_bits(a) -> np.ndarray:
    """fp16 values as their uint16 bit patterns (a view of a contiguous fp16 copy)."""
    return np.ascontiguousarray(a, dtype=np.float16).view(np.uint16)

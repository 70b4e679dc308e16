"""GB300 (sm_103a) prefill of the clef-flash hybrid decoder: thin Python binding of libclef.so.

Every function here only marshals arguments into the C ABI declared in include/clef.h; all of the
computation runs in the library's CUDA kernels.  PyTorch is used for device memory and streams.
There is no fallback: if libclef.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libclef.so")

HIDDEN = 4096
INTER = 12288
GDN_HK, GDN_HV, GDN_D = 16, 32, 128
ATT_HQ, ATT_HKV, ATT_D = 16, 4, 256
MAX_LEN = 16384
SWIGLU_BLOCK = 16

STATUS_NAMES = {
    0: "CLEF_OK", 1: "CLEF_E_INVALID", 2: "CLEF_E_SHAPE", 3: "CLEF_E_TOO_LONG", 4: "CLEF_E_ALIGN",
    5: "CLEF_E_CUDA", 6: "CLEF_E_DEVICE_TIMEOUT", 7: "CLEF_E_NONFINITE", 8: "CLEF_E_WORKSPACE",
    9: "CLEF_E_BAD_TOKEN",
}


class ClefError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}: {msg}")


class Lut6(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("lut", ctypes.c_void_p)]


class Layer(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("attn_norm", ctypes.c_void_p),
        ("mlp_norm", ctypes.c_void_p),
        ("in_proj", Lut6),
        ("out_proj", Lut6),
        ("gate_up", Lut6),
        ("down", Lut6),
        ("ab_w", ctypes.c_void_p),
        ("A_log", ctypes.c_void_p),
        ("dt_bias", ctypes.c_void_p),
        ("conv_w", ctypes.c_void_p),
        ("o_norm", ctypes.c_void_p),
    ]


class Model(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32),
        ("layers", ctypes.POINTER(Layer)),
        ("embed", ctypes.c_void_p),
        ("vocab", ctypes.c_int64),
        ("final_norm", ctypes.c_void_p),
        ("flags", ctypes.c_int32),
    ]


MODEL_REPRODUCIBLE = 1


class State(ctypes.Structure):
    """clef_state: the carried state of a chunked prefill (device buffers, see clef.h)."""
    _fields_ = [
        ("conv", ctypes.c_void_p),
        ("rec", ctypes.c_void_p),
        ("kcache", ctypes.c_void_p),
        ("vcache", ctypes.c_void_p),
        ("ctx", ctypes.c_int64),
        ("pos", ctypes.c_int64),
    ]


_lib = None

_SIGS = {
    "clef_last_error": (ctypes.c_char_p, []),
    "clef_version": (ctypes.c_int32, []),
    "clef_debug_fail_next": (None, [ctypes.c_int32]),
    "clef_debug_gdn_workspace_layout": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                                       ctypes.c_void_p, ctypes.c_void_p]),
    "clef_sync_status": (ctypes.c_int, [ctypes.c_void_p]),
    "clef_check_finite": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p]),
    "clef_lut6_pack": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "clef_lut6_unpack": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "clef_lut6_dequant": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p, ctypes.c_void_p]),
    "clef_lut6_tile": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                      ctypes.c_void_p]),
    "clef_lut6_quantize": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]),
    "clef_lut6_gemm": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_void_p]),
    "clef_lut6_gemm_canonical_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "clef_lut6_gemm_canonical": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int32] + [ctypes.c_int64] * 3 +
                                 [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "clef_gdn_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "clef_gdn_prefill": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_int64, ctypes.c_int64,
                                                                  ctypes.c_void_p, ctypes.c_size_t,
                                                                  ctypes.c_void_p]),
    "clef_gdn_prefill_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_int64, ctypes.c_int64,
                                                                          ctypes.c_void_p]),
    "clef_attn_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "clef_gqa_attn_prefill": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 5 +
                              [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "clef_prefill_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "clef_prefill_forward": (ctypes.c_int, [ctypes.POINTER(Model), ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_size_t, ctypes.c_void_p]),
    "clef_mrope_positions": (ctypes.c_int, [ctypes.c_int64] * 4 + [ctypes.c_void_p]),
    "clef_prefill_forward_image": (ctypes.c_int, [ctypes.POINTER(Model), ctypes.c_void_p, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "clef_prefill_chunk_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "clef_prefill_forward_chunk": (ctypes.c_int, [ctypes.POINTER(Model), ctypes.c_void_p, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.POINTER(State), ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "clef_decoder_layer": (ctypes.c_int, [ctypes.POINTER(Layer), ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                          ctypes.c_void_p]),
}


def lib():
    """The loaded libclef.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name, None)
            if fn is None:
                continue
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(code: int, where: str):
    if code != 0:
        raise ClefError(code, where, lib().clef_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("expected contiguous CUDA tensors")


def sync_status(stream=None):
    """Synchronise the stream and raise if a kernel reported a device-side problem."""
    _check(lib().clef_sync_status(_stream(stream)), "clef_sync_status")


def check_finite(x, stream=None):
    """Device: per-row flags (uint8 [rows], 1 = the row holds an inf or a NaN) of an fp16 tensor
    viewed as [rows, last dim]; a flagged row is also reported to sync_status()."""
    _need_cuda(x)
    if x.dtype != torch.float16 or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp16 CUDA tensor")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    flags = torch.empty(rows, dtype=torch.uint8, device=x.device)
    _check(lib().clef_check_finite(_ptr(x), rows, cols, _ptr(flags), _stream(stream)), "clef_check_finite")
    return flags


# ------------------------------------------------------------------------------------- LUT-6
def lut6_pack(idx):
    """Host: pack uint8 indices [n, k] (numpy or CPU tensor) into [n, k*3/4] bytes."""
    import numpy as np
    a = np.ascontiguousarray(np.asarray(idx, dtype=np.uint8))
    n, k = a.shape
    out = np.empty((n, k * 3 // 4), dtype=np.uint8)
    _check(lib().clef_lut6_pack(a.ctypes.data, n, k, out.ctypes.data), "clef_lut6_pack")
    return out


def mrope_positions(L, image_start=0, grid=(0, 0)):
    """Host: [L, 3] int32 M-RoPE positions (t, h, w) of a request with at most one picture."""
    import numpy as np
    out = np.empty((L, 3), dtype=np.int32)
    _check(lib().clef_mrope_positions(L, image_start, grid[0], grid[1], out.ctypes.data),
           "clef_mrope_positions")
    return out


def lut6_unpack(packed, k):
    import numpy as np
    a = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8))
    n = a.shape[0]
    out = np.empty((n, k), dtype=np.uint8)
    _check(lib().clef_lut6_unpack(a.ctypes.data, n, k, out.ctypes.data), "clef_lut6_unpack")
    return out


def lut6_dequant(packed, lut, k, stream=None):
    """Device: dense fp16 W [n, k] from a LUT-6 weight."""
    _need_cuda(packed, lut)
    n = lut.shape[0] * 16
    w = torch.empty((n, k), dtype=torch.float16, device=packed.device)
    _check(lib().clef_lut6_dequant(_ptr(packed), _ptr(lut), n, k, _ptr(w), _stream(stream)),
           "clef_lut6_dequant")
    return w


def lut6_tile(packed, k, stream=None):
    """Device: the GEMM's tiled layout of a canonical packed LUT-6 weight [n, k*3/4]."""
    _need_cuda(packed)
    n = packed.shape[0]
    tiled = torch.empty_like(packed)
    _check(lib().clef_lut6_tile(_ptr(packed), n, k, _ptr(tiled), _stream(stream)), "clef_lut6_tile")
    return tiled


def lut6_quantize(w, stream=None):
    """Device: LUT-6 quantisation of an fp16 weight w [n, k] -> (packed [n, k*3/4] uint8 in the
    canonical row-major layout, lut [n/16, 64] fp16)."""
    _need_cuda(w)
    if w.dtype != torch.float16 or w.dim() != 2:
        raise ValueError("w must be a 2-D fp16 tensor")
    w = w.contiguous()
    n, k = w.shape
    packed = torch.empty((n, k * 3 // 4), dtype=torch.uint8, device=w.device)
    lut = torch.empty((n // 16, 64), dtype=torch.float16, device=w.device)
    _check(lib().clef_lut6_quantize(_ptr(w), n, k, _ptr(packed), _ptr(lut), _stream(stream)),
           "clef_lut6_quantize")
    return packed, lut


def lut6_gemm(x, packed, lut, out_fp32=False, out=None, stream=None, tiled=False):
    """Device: y = x . W^T for fp16 x [m, k] and LUT-6 W [n, k]; y fp16 (or fp32) [m, n].

    `packed` is the canonical [n, k*3/4] stream (clef_lut6_gemm_canonical, which tiles it into a
    workspace first), or (tiled=True) already in the GEMM layout of lut6_tile (clef_lut6_gemm)."""
    _need_cuda(x, packed, lut)
    m, k = x.shape
    n = lut.shape[0] * 16
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32 if out_fp32 else torch.float16, device=x.device)
    if tiled:
        _check(lib().clef_lut6_gemm(_ptr(x), _ptr(packed), _ptr(lut), _ptr(out), 1 if out_fp32 else 0,
                                    m, n, k, _stream(stream)), "clef_lut6_gemm")
    else:
        ws = _workspace(lib().clef_lut6_gemm_canonical_workspace_size(n, k), x.device)
        _check(lib().clef_lut6_gemm_canonical(_ptr(x), _ptr(packed), _ptr(lut), _ptr(out),
                                              1 if out_fp32 else 0, m, n, k, _ptr(ws), ws.numel(),
                                              _stream(stream)), "clef_lut6_gemm_canonical")
    return out


# --------------------------------------------------------------------------- GDN and attention
def _workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def gdn_prefill(q, k, v, alpha, beta, s0=None, want_state=False, stream=None):
    """Device: the gated delta rule over B requests of L positions.

    q, k [B, L, 16, 128] fp16; v [B, L, 32, 128] fp16; alpha, beta [B, L, 32] fp32;
    s0 [B, 32, 128, 128] fp32 or None.  Returns o [B, L, 32, 128] fp16 (and S_L if want_state).
    """
    _need_cuda(q, k, v, alpha, beta, s0)
    B, L = q.shape[0], q.shape[1]
    o = torch.empty((B, L, GDN_HV, GDN_D), dtype=torch.float16, device=q.device)
    s_out = torch.empty((B, GDN_HV, GDN_D, GDN_D), dtype=torch.float32, device=q.device) if want_state else None
    ws = _workspace(lib().clef_gdn_workspace_size(B, L), q.device)
    _check(lib().clef_gdn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(s0), _ptr(o),
                                  _ptr(s_out), B, L, _ptr(ws), ws.numel(), _stream(stream)),
           "clef_gdn_prefill")
    return (o, s_out) if want_state else o


def gqa_attn_prefill(q, k, v, gate=None, stream=None):
    """Device: causal GQA attention with rotary; q [B, L, 16, 256], k, v [B, L, 4, 256] fp16,
    gate [B, L, 16, 256] fp16 or None.  Returns o [B, L, 16, 256] fp16."""
    _need_cuda(q, k, v, gate)
    B, L = q.shape[0], q.shape[1]
    o = torch.empty((B, L, ATT_HQ, ATT_D), dtype=torch.float16, device=q.device)
    ws = _workspace(lib().clef_attn_workspace_size(B, L), q.device)
    _check(lib().clef_gqa_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(o), B, L, 0, 0, 0,
                                       _ptr(ws), ws.numel(), _stream(stream)), "clef_gqa_attn_prefill")
    return o


def prefill_workspace_size(B, L):
    return int(lib().clef_prefill_workspace_size(B, L))


def decoder_layer(layer, x, workspace=None, stream=None):
    """Device: one decoder layer on the fp32 residual stream x [B, L, 4096], in place."""
    _need_cuda(x)
    B, L = x.shape[0], x.shape[1]
    ws = workspace if workspace is not None else _workspace(prefill_workspace_size(B, L), x.device)
    _check(lib().clef_decoder_layer(ctypes.byref(layer.struct), _ptr(x), B, L, _ptr(ws), ws.numel(),
                                    _stream(stream)), "clef_decoder_layer")
    return x

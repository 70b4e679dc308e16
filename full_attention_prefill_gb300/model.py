"""Device-resident clef-flash weights in the library's layout, and the prefill call.

The layout is the C ABI's (include/clef.h, clef_layer / clef_model): per layer one fused input
projection (GDN: q | k | v | z rows; attention: query | gate | k | v rows), the output
projection, the MLP gate and up rows interleaved in blocks of 64, and the down projection, all
LUT-6 in the GEMM's tiled layout (clef_lut6_tile); GDN small weights fp16.  Building a layer only
moves bytes (row blocks of the packed indices and their tables are concatenated or interleaved,
then the quadruples are tiled); no weight value changes.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import (HIDDEN, SWIGLU_BLOCK, Layer, Lut6, Model, State, _check, _ptr, _stream, _workspace,
               lib, lut6_tile, prefill_workspace_size)

GDN, ATTENTION = 0, 1


def _cat_lut6(parts):
    packed = np.concatenate([p for p, _ in parts], axis=0)
    lut = np.concatenate([t for _, t in parts], axis=0)
    return packed, lut


def interleave_gate_up(gate, up, block=SWIGLU_BLOCK):
    """Rows [2jb, 2jb+b) = gate rows [jb, jb+b), rows [2jb+b, 2jb+2b) = up rows [jb, jb+b)."""
    gp, gl = gate
    upk, ul = up
    n = gp.shape[0]
    assert n % block == 0 and upk.shape[0] == n
    nb = n // block
    packed = np.stack([gp.reshape(nb, block, -1), upk.reshape(nb, block, -1)], axis=1).reshape(2 * n, -1)
    tb = block // 16
    lut = np.stack([gl.reshape(nb, tb, 64), ul.reshape(nb, tb, 64)], axis=1).reshape(2 * n // 16, 64)
    return packed, lut


class DeviceLayer:
    """One decoder layer's weights on the device plus its clef_layer struct."""

    def __init__(self, w: dict, kind: int, device="cuda"):
        self.kind = kind
        self._keep = []

        def dev(a):
            t = torch.from_numpy(np.ascontiguousarray(a)).to(device)
            self._keep.append(t)
            return t

        def lut6(pair):
            packed, lut = pair
            k = packed.shape[1] * 4 // 3
            canon = torch.from_numpy(np.ascontiguousarray(packed)).to(device)
            tiled = lut6_tile(canon, k)      # the GEMM's operand layout (same bytes, moved)
            self._keep.append(tiled)
            del canon
            return Lut6(_ptr(tiled), _ptr(dev(lut)))

        st = Layer()
        st.kind = kind
        st.attn_norm = _ptr(dev(w["attn_norm"]))
        st.mlp_norm = _ptr(dev(w["mlp_norm"]))
        if kind == GDN:
            st.in_proj = lut6(_cat_lut6([w["qkv"], w["z"]]))
            st.out_proj = lut6(w["out"])
            st.ab_w = _ptr(dev(np.concatenate([w["a_w"], w["b_w"]], axis=0)))
            st.A_log = _ptr(dev(w["A_log"]))
            st.dt_bias = _ptr(dev(w["dt_bias"]))
            st.conv_w = _ptr(dev(w["conv_w"]))
            st.o_norm = _ptr(dev(w["o_norm"]))
        else:
            st.in_proj = lut6(_cat_lut6([w["q"], w["k"], w["v"]]))
            st.out_proj = lut6(w["o"])
        st.gate_up = lut6(interleave_gate_up(w["gate"], w["up"]))
        st.down = lut6(w["down"])
        self.struct = st

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in self._keep)


class DeviceModel:
    """The hybrid decoder on the device: layers, embedding table, final norm."""

    def __init__(self, layers, embed, final_norm, device="cuda"):
        self.layers = layers
        if isinstance(embed, np.ndarray):
            embed = torch.from_numpy(np.ascontiguousarray(embed)).to(device)
        self.embed = embed
        self.final_norm = torch.from_numpy(np.ascontiguousarray(final_norm)).to(device)
        arr = (Layer * len(layers))(*[l.struct for l in layers])
        self._arr = arr
        m = Model()
        m.n_layers = len(layers)
        m.layers = ctypes.cast(arr, ctypes.POINTER(Layer))
        m.embed = _ptr(self.embed)
        m.vocab = self.embed.shape[0]
        m.final_norm = _ptr(self.final_norm)
        m.flags = 0
        self.struct = m
        self._ws = None

    def set_reproducible(self, on: bool = True):
        """Ordered reduction of split residual adds (clef.h CLEF_MODEL_REPRODUCIBLE): every run of
        the same prefill then gives the same bits."""
        self.struct.flags = 1 if on else 0

    @staticmethod
    def kind_of(layer_index: int) -> int:
        return ATTENTION if layer_index % 4 == 3 else GDN

    def workspace(self, B, L):
        need = prefill_workspace_size(B, L)
        if self._ws is None or self._ws.numel() < need:
            self._ws = None
            self._ws = _workspace(need, self.embed.device)
        return self._ws

    def forward(self, ids, out=None, stream=None):
        """ids [B, L] int32 (device) -> final-norm hidden [B, L, 4096] fp16."""
        if not (ids.is_cuda and ids.dtype == torch.int32 and ids.is_contiguous()):
            raise ValueError("ids must be a contiguous int32 CUDA tensor")
        B, L = ids.shape
        if out is None:
            out = torch.empty((B, L, HIDDEN), dtype=torch.float16, device=ids.device)
        ws = self.workspace(B, L)
        _check(lib().clef_prefill_forward(ctypes.byref(self.struct), _ptr(ids), B, L, _ptr(out), _ptr(ws),
                                          ws.numel(), _stream(stream)), "clef_prefill_forward")
        return out

    def forward_image(self, ids, image_rows, image_start, grid, out=None, stream=None):
        """ids [B, L] int32 (device) with a picture block of grid = (H, W) tokens at image_start
        in every request; image_rows [B, H*W, 4096] fp16 (device) -> hidden [B, L, 4096] fp16
        (M-RoPE positions in the attention layers)."""
        if not (ids.is_cuda and ids.dtype == torch.int32 and ids.is_contiguous()):
            raise ValueError("ids must be a contiguous int32 CUDA tensor")
        B, L = ids.shape
        n = grid[0] * grid[1]
        if n and not (image_rows.is_cuda and image_rows.dtype == torch.float16 and
                      tuple(image_rows.shape) == (B, n, HIDDEN) and image_rows.is_contiguous()):
            raise ValueError("image_rows must be a contiguous fp16 CUDA tensor [B, H*W, 4096]")
        if out is None:
            out = torch.empty((B, L, HIDDEN), dtype=torch.float16, device=ids.device)
        ws = self.workspace(B, L)
        _check(lib().clef_prefill_forward_image(ctypes.byref(self.struct), _ptr(ids), B, L,
                                                _ptr(image_rows) if n else None, image_start,
                                                grid[0], grid[1], _ptr(out), _ptr(ws), ws.numel(),
                                                _stream(stream)), "clef_prefill_forward_image")
        return out

    def forward_chunk(self, ids, state, out=None, stream=None):
        """ids [B, L] int32 (device): positions state.pos .. state.pos + L - 1 of the state's
        requests -> their final-norm hidden [B, L, 4096] fp16; the state moves on by L."""
        if not (ids.is_cuda and ids.dtype == torch.int32 and ids.is_contiguous()):
            raise ValueError("ids must be a contiguous int32 CUDA tensor")
        B, L = ids.shape
        if B != state.B:
            raise ValueError(f"ids carry {B} requests, the state {state.B}")
        if out is None:
            out = torch.empty((B, L, HIDDEN), dtype=torch.float16, device=ids.device)
        ws = self.workspace(B, L)
        _check(lib().clef_prefill_forward_chunk(ctypes.byref(self.struct), _ptr(ids), B, L,
                                                ctypes.byref(state.struct), _ptr(out), _ptr(ws), ws.numel(),
                                                _stream(stream)), "clef_prefill_forward_chunk")
        return out


class PrefillState:
    """The carried state of B requests for DeviceModel.forward_chunk: torch-allocated, zeroed
    (an empty state), in the layouts of clef_state."""

    def __init__(self, model, B, ctx, device="cuda"):
        n_gdn = sum(1 for l in model.layers if l.kind == GDN)
        n_attn = len(model.layers) - n_gdn
        self.conv = torch.zeros((max(n_gdn, 1), B, 3, 8192), dtype=torch.float16, device=device)
        self.rec = torch.zeros((max(n_gdn, 1), B, 32, 128, 128), dtype=torch.float32, device=device)
        self.kcache = torch.zeros((max(n_attn, 1), B, ctx, 4, 256), dtype=torch.float16, device=device)
        self.vcache = torch.zeros_like(self.kcache)
        st = State()
        st.conv, st.rec = _ptr(self.conv), _ptr(self.rec)
        st.kcache, st.vcache = _ptr(self.kcache), _ptr(self.vcache)
        st.ctx, st.pos = ctx, 0
        self.struct = st
        self.B = B

    @property
    def pos(self):
        return self.struct.pos

    def clone(self):
        """An independent copy (device-to-device) at the same position: a shared part prefilled
        once can then be continued by several question parts, each on its own copy."""
        c = PrefillState.__new__(PrefillState)
        c.conv, c.rec = self.conv.clone(), self.rec.clone()
        c.kcache, c.vcache = self.kcache.clone(), self.vcache.clone()
        st = State()
        st.conv, st.rec = _ptr(c.conv), _ptr(c.rec)
        st.kcache, st.vcache = _ptr(c.kcache), _ptr(c.vcache)
        st.ctx, st.pos = self.struct.ctx, self.struct.pos
        c.struct = st
        c.B = self.B
        return c


def synth_model(seed=0, n_layers=32, device="cuda", embed=None):
    """The synthetic model (seeded random weights, the recipe of the `synth` module)."""
    import synth
    layers = []
    for l in range(n_layers):
        kind = DeviceModel.kind_of(l)
        layers.append(DeviceLayer(synth.layer_weights(seed, l), kind, device))
    if embed is None:
        embed = synth.embedding_table(seed)
    return DeviceModel(layers, embed, synth.final_norm_weight(seed), device)

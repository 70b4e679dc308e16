"""The joint schema head on the device: weights in the C ABI's struct (clef_head) and the call.

Only moves bytes and marshals arguments into clef_joint_head (include/clef.h, which states what
the pages fix about the head and the reading taken for its layers).
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _check, _need_cuda, _ptr, _stream, _workspace, lib

_LAYER_NAMES = ("norm1", "wq", "wk", "wv", "wo", "norm2", "wg", "wu", "wd")
_TOP_NAMES = ("w_mem", "w_in", "w_lex", "e_qtype", "e_opt", "e_glob")


class HeadLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LAYER_NAMES]


class Head(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_void_p) for n in _TOP_NAMES] +
                [("dec", HeadLayer * 4), ("route", HeadLayer * 2)] +
                [(n, ctypes.c_void_p) for n in ("norm_f", "w_opt", "w_qst")])


_sigs_set = False


def _sigs():
    global _sigs_set
    if _sigs_set:
        return
    L = lib()
    L.clef_joint_head_workspace_size.restype = ctypes.c_size_t
    L.clef_joint_head_workspace_size.argtypes = [ctypes.c_int64] * 3
    L.clef_joint_head.restype = ctypes.c_int
    L.clef_joint_head.argtypes = ([ctypes.POINTER(Head), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64] +
                                  [ctypes.c_void_p] * 8 + [ctypes.c_int64, ctypes.c_int64] +
                                  [ctypes.c_void_p] * 3 + [ctypes.c_size_t, ctypes.c_void_p])
    _sigs_set = True


class DeviceHead:
    """The head's fp16 weights on the device (a dict of the synth recipe's names)."""

    def __init__(self, w: dict, device="cuda"):
        self._keep = []

        def dev(a):
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(device)
            self._keep.append(t)
            return _ptr(t)

        h = Head()
        for n in _TOP_NAMES + ("norm_f", "w_opt", "w_qst"):
            setattr(h, n, dev(w[n]))
        for kind, count in (("dec", 4), ("route", 2)):
            for i in range(count):
                layer = getattr(h, kind)[i]
                for n in _LAYER_NAMES:
                    setattr(layer, n, dev(w[kind][i][n]))
        self.struct = h

    def __call__(self, hidden, q_avg, o_avg, g_avg, lexical, member, type_ids, q_valid=None,
                 o_valid=None, key_valid=None, stream=None):
        """hidden [T, 4096] fp16 (device); the rest device tensors (fp32 spans and lexical rows,
        uint8 member / validity, int32 type ids).  Returns (logits [O], probs [O]) fp32."""
        _sigs()
        _need_cuda(hidden, q_avg, o_avg, g_avg, lexical, member, type_ids)
        dev = hidden.device
        T, Q, O = hidden.shape[0], q_avg.shape[0], o_avg.shape[0]
        ones = lambda n: torch.ones(n, dtype=torch.uint8, device=dev)  # noqa: E731
        q_valid = ones(Q) if q_valid is None else q_valid
        o_valid = ones(O) if o_valid is None else o_valid
        key_valid = ones(T) if key_valid is None else key_valid
        logits = torch.empty(O, dtype=torch.float32, device=dev)
        probs = torch.empty(O, dtype=torch.float32, device=dev)
        ws = _workspace(lib().clef_joint_head_workspace_size(T, Q, O), dev)
        _check(lib().clef_joint_head(ctypes.byref(self.struct), _ptr(hidden), _ptr(key_valid), T, _ptr(q_avg),
                                     _ptr(o_avg), _ptr(g_avg), _ptr(lexical), _ptr(member), _ptr(type_ids),
                                     _ptr(q_valid), _ptr(o_valid), Q, O, _ptr(logits), _ptr(probs),
                                     _ptr(ws), ws.numel(), _stream(stream)), "clef_joint_head")
        return logits, probs

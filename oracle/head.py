"""The joint schema head, oracle side: thin marshalling over the C++ oracle (oracle/csrc/head.cpp,
which states what the pages fix about the head and the reading taken for its layers).
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import check, contig, f16_bits, f64, lib, ptr


class HeadLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("norm1", "wq", "wk", "wv", "wo", "norm2", "wg", "wu", "wd")]


class Head(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_void_p) for n in ("w_mem", "w_in", "w_lex", "e_qtype", "e_opt", "e_glob")] +
                [("dec", HeadLayer * 4), ("route", HeadLayer * 2)] +
                [(n, ctypes.c_void_p) for n in ("norm_f", "w_opt", "w_qst")])


def _head_struct(w, keep):
    h = Head()

    def bits(a):
        b = f16_bits(a)
        keep.append(b)
        return b.ctypes.data

    for n in ("w_mem", "w_in", "w_lex", "e_qtype", "e_opt", "e_glob", "norm_f", "w_opt", "w_qst"):
        setattr(h, n, bits(w[n]))
    for kind, count in (("dec", 4), ("route", 2)):
        for i in range(count):
            layer = getattr(h, kind)[i]
            for n, _ in HeadLayer._fields_:
                setattr(layer, n, bits(w[kind][i][n]))
    return h


def joint_head(hidden, w, q_avg, o_avg, g_avg, lexical, member, type_ids, q_valid=None,
               o_valid=None, key_valid=None):
    """hidden [T, 4096] -> (logits [O], probs [O]) in float64."""
    H = f64(hidden)
    T = H.shape[0]
    qa, oa, ga, lex = f64(q_avg), f64(o_avg), f64(g_avg).reshape(T), f64(lexical)
    Q, O = qa.shape[0], oa.shape[0]
    mem = contig(member, np.uint8)
    tid = contig(type_ids, np.int32)
    qv = contig(np.ones(Q) if q_valid is None else q_valid, np.uint8)
    ov = contig(np.ones(O) if o_valid is None else o_valid, np.uint8)
    kv = contig(np.ones(T) if key_valid is None else key_valid, np.uint8)
    keep = []
    hs = _head_struct(w, keep)
    logits, probs = np.empty(O), np.empty(O)
    check(lib().orc_joint_head(ptr(H), ptr(kv), T, ptr(qa), ptr(oa), ptr(ga), ptr(lex), ptr(mem),
                               ptr(tid), ptr(qv), ptr(ov), Q, O, ctypes.byref(hs), ptr(logits),
                               ptr(probs)), "joint_head")
    return logits, probs

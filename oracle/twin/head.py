"""The joint schema head: the numpy twin of the C++ oracle (float64).  The same definition as
oracle/csrc/head.cpp (which states what the pages fix and the reading taken for the layers),
written independently with numpy matrix products."""
from __future__ import annotations

import numpy as np

D, NH, DH = 1024, 16, 64


def _f(a):
    return np.asarray(a, dtype=np.float64)


def _rms(x, w):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6) * _f(w)


def _attend(q, k, v, valid):
    S, T = q.shape[0], k.shape[0]
    out = np.zeros((S, D))
    if not np.any(valid):
        return out
    qh = q.reshape(S, NH, DH).transpose(1, 0, 2)
    kh = k.reshape(T, NH, DH).transpose(1, 0, 2)
    vh = v.reshape(T, NH, DH).transpose(1, 0, 2)
    logits = qh @ kh.transpose(0, 2, 1) / np.sqrt(DH)            # [NH, S, T]
    logits = np.where(np.asarray(valid, bool)[None, None, :], logits, -np.inf)
    p = np.exp(logits - logits.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    return (p @ vh).transpose(1, 0, 2).reshape(S, D)


def _layer(s, L, mem, mem_valid, slot_valid):
    a = _rms(s, L["norm1"])
    src = a if mem is None else mem
    o = _attend(a @ _f(L["wq"]).T, src @ _f(L["wk"]).T, src @ _f(L["wv"]).T,
                slot_valid if mem is None else mem_valid)
    s = s + o @ _f(L["wo"]).T
    b = _rms(s, L["norm2"])
    g = b @ _f(L["wg"]).T
    return s + ((g / (1 + np.exp(-g))) * (b @ _f(L["wu"]).T)) @ _f(L["wd"]).T


def joint_head(hidden, w, q_avg, o_avg, g_avg, lexical, member, type_ids, q_valid=None,
               o_valid=None, key_valid=None):
    H = _f(hidden)
    T = H.shape[0]
    Q, O = np.shape(q_avg)[0], np.shape(o_avg)[0]
    qv = np.ones(Q, bool) if q_valid is None else np.asarray(q_valid, bool)
    ov = np.ones(O, bool) if o_valid is None else np.asarray(o_valid, bool)
    kv = np.ones(T, bool) if key_valid is None else np.asarray(key_valid, bool)
    u = np.concatenate([_f(q_avg), _f(o_avg), _f(g_avg).reshape(1, T)]) @ H
    s = u @ _f(w["w_in"]).T
    s[:Q] += _f(w["e_qtype"])[np.asarray(type_ids)]
    s[Q:Q + O] += _f(lexical) @ _f(w["w_lex"]).T + _f(w["e_opt"])
    s[Q + O] += _f(w["e_glob"])
    mem = H @ _f(w["w_mem"]).T
    slot_valid = np.concatenate([qv, ov, [True]])
    for L in w["dec"]:
        s = _layer(s, L, mem, kv, None)
    for L in w["route"]:
        s = _layer(s, L, None, None, slot_valid)
    f = _rms(s, w["norm_f"])
    c = np.asarray(member, np.float64).T @ f[:Q]                  # [O, D]
    logits = np.sum((f[Q:Q + O] @ _f(w["w_opt"]).T) * (c @ _f(w["w_qst"]).T), axis=1) / np.sqrt(D)
    logits = np.where(ov, logits, 0.0)
    probs = np.zeros(O)
    for q in range(Q):
        sel = np.asarray(member[q], bool) & ov
        if qv[q] and sel.any():
            z = np.exp(logits[sel] - logits[sel].max())
            probs[sel] = z / z.sum()
    return logits, probs

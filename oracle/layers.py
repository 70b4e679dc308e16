"""Oracle building blocks of the clef-flash decoder layers: thin marshalling over the C++ oracle
(oracle/csrc/layers.cpp, fp64).  Each C++ function states the passage it follows; the readings
(eps, scales, head maps, rotary pairing, M-RoPE planes) are stated there.
"""
from __future__ import annotations

import numpy as np

from ._lib import check, contig, f64, lib, ptr

RMS_EPS = 1e-6
L2_EPS = 1e-6
ROPE_THETA = 1.0e7
ROPE_DIMS = 64
MROPE_SECTIONS = (11, 11, 10)   # frequency pairs on the t, h and w planes


def _elementwise(fn, x):
    xx = f64(x)
    out = np.empty_like(xx)
    fn(ptr(xx), xx.size, ptr(out))
    return out


def silu(x):
    return _elementwise(lib().orc_silu, x)


def sigmoid(x):
    return _elementwise(lib().orc_sigmoid, x)


def softplus(x):
    return _elementwise(lib().orc_softplus, x)


def rmsnorm(x, w, eps=RMS_EPS):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w."""
    xx = f64(x)
    d = xx.shape[-1]
    ww = np.broadcast_to(f64(w), (d,)).copy() if w is not None else None
    out = np.empty_like(xx)
    lib().orc_rmsnorm(ptr(xx), xx.size // d if d else 0, d, ptr(ww), float(eps), ptr(out))
    return out


def l2norm(x, eps=L2_EPS):
    """x / sqrt(sum(x^2) + eps) over the last axis."""
    xx = f64(x)
    d = xx.shape[-1]
    out = np.empty_like(xx)
    lib().orc_l2norm(ptr(xx), xx.size // d if d else 0, d, float(eps), ptr(out))
    return out


def causal_conv_silu(x, w):
    """Causal depthwise conv (zero history) then SiLU.  x: [L, C], w: [C, taps]."""
    xx, ww = f64(x), f64(w)
    L, C = xx.shape
    out = np.empty_like(xx)
    lib().orc_conv_silu(ptr(xx), L, C, ptr(ww), ww.shape[1], ptr(out))
    return out


def gdn_gates(a, b, A_log, dt_bias):
    """alpha = exp(-exp(A_log) softplus(a + dt_bias)), beta = sigmoid(b); a, b [L, Hv]."""
    aa, bb = f64(a), f64(b)
    L, H = aa.shape
    A, dt = f64(np.broadcast_to(f64(A_log), (H,))), f64(np.broadcast_to(f64(dt_bias), (H,)))
    alpha, beta = np.empty_like(aa), np.empty_like(aa)
    lib().orc_gdn_gates(ptr(aa), ptr(bb), L, H, ptr(A), ptr(dt), ptr(alpha), ptr(beta))
    return alpha, beta


def gated_delta_rule(q, k, v, alpha, beta, s0=None):
    """The per-token gated delta rule.  q, k: [L, Hk, dk]; v: [L, Hv, dv]; alpha, beta: [L, Hv];
    s0 [Hv, dv, dk] or None.  Returns (o [L, Hv, dv], S_L [Hv, dv, dk])."""
    qq, kk, vv = f64(q), f64(k), f64(v)
    aa, bb = f64(alpha), f64(beta)
    L, Hk, dk = kk.shape
    Hv, dv = vv.shape[1], vv.shape[2]
    ss = None if s0 is None else f64(s0)
    o = np.empty((L, Hv, dv))
    S = np.empty((Hv, dv, dk))
    check(lib().orc_gated_delta_rule(ptr(qq), ptr(kk), ptr(vv), ptr(aa), ptr(bb), ptr(ss), L, Hk, Hv,
                                     dk, dv, ptr(o), ptr(S)), "gated_delta_rule")
    return o, S


def zgated_norm(o, z, w, eps=RMS_EPS):
    """RMSNorm over each head's dv values, times w, times SiLU(z).  o, z: [L, Hv, dv] -> [L, Hv*dv]."""
    oo, zz, ww = f64(o), f64(z), f64(w)
    L, H, d = oo.shape
    out = np.empty_like(oo)
    lib().orc_zgated_norm(ptr(oo), ptr(zz), L, H, d, ptr(ww), float(eps), ptr(out))
    return out.reshape(L, H * d)


def rope(x, positions, rot_dims=ROPE_DIMS, theta=ROPE_THETA):
    """1-D rotary on the first `rot_dims` dims of each head.  x: [L, H, D]; positions: [L]."""
    xx = f64(x)
    L, H, D = xx.shape
    pos = f64(positions).reshape(L)
    out = np.empty_like(xx)
    lib().orc_rope(ptr(xx), L, H, D, ptr(pos), rot_dims, float(theta), ptr(out))
    return out


def mrope_planes(rot_dims=ROPE_DIMS):
    """Plane (0 = t, 1 = h, 2 = w) of each of the rot_dims / 2 frequency pairs."""
    out = np.empty(rot_dims // 2, dtype=np.int64)
    lib().orc_mrope_planes(rot_dims, ptr(out))
    return out


def mrope_positions(L, image_start=0, grid_h=0, grid_w=0):
    """[L, 3] integer positions (t, h, w) of a request holding at most one picture block."""
    out = np.empty((L, 3), dtype=np.int64)
    check(lib().orc_mrope_positions(L, image_start, grid_h, grid_w, ptr(out)), "mrope_positions")
    return out


def mrope(x, pos3, rot_dims=ROPE_DIMS, theta=ROPE_THETA):
    """Multimodal rotary: pair j turns by pos3[:, plane(j)] * theta^(-2j/64)."""
    xx = f64(x)
    L, H, D = xx.shape
    p3 = contig(pos3, np.int64).reshape(L, 3)
    out = np.empty_like(xx)
    lib().orc_mrope(ptr(xx), L, H, D, ptr(p3), rot_dims, float(theta), ptr(out))
    return out


def causal_attention(q, k, v, rows=None):
    """Causal GQA softmax attention, one explicit softmax per query row.
    q: [L, Hq, D]; k, v: [L, Hkv, D].  Returns [L, Hq, D], or only query rows r0 .. r1 - 1 when
    rows = (r0, r1)."""
    qq, kk, vv = f64(q), f64(k), f64(v)
    L, Hq, D = qq.shape
    Hkv = kk.shape[1]
    r0, r1 = (0, L) if rows is None else rows
    out = np.empty((r1 - r0, Hq, D))
    check(lib().orc_causal_attention(ptr(qq), ptr(kk), ptr(vv), L, Hq, Hkv, D, r0, r1, ptr(out)),
          "causal_attention")
    return out

"""Oracle building blocks of the decoder layers: the numpy twin of the C++ oracle (float64).

Each function states the passage it follows.  Shapes use L = positions of one request.
Where a page is silent the plainest reading is taken and named in the docstring.
"""
from __future__ import annotations

import numpy as np

RMS_EPS = 1e-6
L2_EPS = 1e-6
ROPE_THETA = 1.0e7
ROPE_DIMS = 64


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def silu(x):
    x = f64(x)
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    x = f64(x)
    return 1.0 / (1.0 + np.exp(-x))


def softplus(x):
    x = f64(x)
    return np.logaddexp(0.0, x)


def rmsnorm(x, w, eps=RMS_EPS):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w.

    "Clef-Flash-ANE-LUT6" §Weight precision lists normalization weights among the FP16 text
    weights; "clef-flash-LiteRT" §Host contract step 6 returns the output of the final
    RMSNorm.  eps = 1e-6 and the plain x * r * w form are the adopted reading (no page gives them).
    """
    x = f64(x)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * f64(w)


def l2norm(x, eps=L2_EPS):
    """x / sqrt(sum(x^2) + eps) over the last axis (per-head q/k normalisation of the GDN)."""
    x = f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def causal_conv_silu(x, w):
    """Short causal depthwise convolution (kernel 4) followed by SiLU.

    "Clef-Flash-ANE-LUT6" §Weight precision names the short convolution; "clef-flash - Core AI"
    §Core AI shape carries a conv state [24, 1, 8192, 3] per GDN layer, i.e. 8,192 channels and a
    kernel of 3 + 1 = 4.  c[t, ch] = SiLU(sum_{j=0..3} w[ch, j] * x[t - 3 + j, ch]), with zero
    history before position 0 (a prefill starts from a zeroed state).
    x: [L, C], w: [C, 4].
    """
    x = f64(x)
    w = f64(w)
    L, C = x.shape
    ksz = w.shape[1]
    acc = np.zeros((L, C))
    for j in range(ksz):
        shift = ksz - 1 - j              # tap j reads position t - shift
        if shift == 0:
            acc += w[:, j] * x
        elif shift < L:
            acc[shift:] += w[:, j] * x[: L - shift]
    return silu(acc)


def gdn_gates(a, b, A_log, dt_bias):
    """Per-value-head decay and write strength of the Gated DeltaNet.

    "Clef-Flash-ANE-LUT6" §Weight precision keeps the gates' projection weights and the decay
    parameters in FP16.  Adopted reading (standard Gated DeltaNet gating):
      alpha = exp(-exp(A_log) * softplus(a + dt_bias)),  beta = sigmoid(b).
    a, b: [L, Hv];  A_log, dt_bias: [Hv].
    """
    alpha = np.exp(-np.exp(f64(A_log)) * softplus(f64(a) + f64(dt_bias)))
    beta = sigmoid(b)
    return alpha, beta


def gated_delta_rule(q, k, v, alpha, beta, s0=None):
    """The gated delta rule as a per-token recurrence (no chunking).

    "Clef-Flash-ANE-LUT6" §Model architecture: 24 Gated DeltaNet layers with 16 key and 32 value
    heads of size 128; "clef-flash - Core AI" §Core AI shape: recurrent state [.., 32, 128, 128]
    per layer, the recurrence unrolled over positions.  For value head h (key head h // 2):
        S_t = alpha_t * S_{t-1} + beta_t * (v_t - alpha_t * S_{t-1} k_t) k_t^T
        o_t = S_t q_t / sqrt(d_k)
    S is [d_v, d_k], S_0 = s0 (zero by default).  The output is read from the updated state and
    scaled by 1/sqrt(d_k) (adopted reading).
    q, k: [L, Hk, dk]; v: [L, Hv, dv]; alpha, beta: [L, Hv].  Returns (o [L, Hv, dv], S_L).
    """
    q, k, v = f64(q), f64(k), f64(v)
    alpha, beta = f64(alpha), f64(beta)
    L, Hk, dk = k.shape
    Hv, dv = v.shape[1], v.shape[2]
    rep = Hv // Hk
    S = np.zeros((Hv, dv, dk)) if s0 is None else f64(s0).copy()
    o = np.empty((L, Hv, dv))
    scale = 1.0 / np.sqrt(dk)
    for t in range(L):
        kt = np.repeat(k[t], rep, axis=0)            # [Hv, dk]
        qt = np.repeat(q[t], rep, axis=0)
        a = alpha[t][:, None, None]
        Sk = np.einsum("hij,hj->hi", S, kt)          # S_{t-1} k_t  [Hv, dv]
        u = beta[t][:, None] * (v[t] - alpha[t][:, None] * Sk)
        S = a * S + u[:, :, None] * kt[:, None, :]
        o[t] = np.einsum("hij,hj->hi", S, qt) * scale
    return o, S


def zgated_norm(o, z, w, eps=RMS_EPS):
    """Output gate of the GDN mixer: RMSNorm over each head's d_v values, times w, times SiLU(z).

    o, z: [L, Hv, dv]; w: [dv] shared by the heads.  Returns [L, Hv * dv].
    """
    y = rmsnorm(o, w, eps) * silu(z)
    return y.reshape(o.shape[0], -1)


def rope(x, positions, rot_dims=ROPE_DIMS, theta=ROPE_THETA):
    """Rotary embedding on the first `rot_dims` dims of each head (rotate-half pairing).

    "clef-flash-coreml" README: decoder parts take cos/sin [L, 64]; "clef-flash-LiteRT" §Host
    contract step 5: theta = 1e7 and text tokens sit at (i, i, i) for their index i, so the three
    M-RoPE planes collapse to one 1-D rotary.  Pairs (j, j + 32) for j < 32 rotate by angle
    pos * theta^(-2j/64); dims 64.. pass through.  x: [L, H, D]; positions: [L].
    """
    x = f64(x).copy()
    half = rot_dims // 2
    inv_freq = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / rot_dims)
    ang = f64(positions)[:, None] * inv_freq[None, :]          # [L, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1 = x[..., :half].copy()
    x2 = x[..., half:rot_dims].copy()
    x[..., :half] = x1 * c - x2 * s
    x[..., half:rot_dims] = x2 * c + x1 * s
    return x


MROPE_SECTIONS = (11, 11, 10)   # frequency pairs on the t, h and w planes


def mrope_planes(rot_dims=ROPE_DIMS):
    """Plane (0 = t, 1 = h, 2 = w) of each of the 32 frequency pairs.

    "clef-flash-LiteRT" §Host contract step 5: three planes, sections 11 / 11 / 10, interleaved.
    Reading: pair j takes plane j mod 3, which gives exactly 11, 11 and 10 pairs.
    """
    return np.arange(rot_dims // 2) % 3


def mrope_positions(L, image_start=0, grid_h=0, grid_w=0):
    """[L, 3] integer positions (t, h, w) of a request holding at most one picture block.

    "clef-flash-LiteRT" §Host contract step 5: text tokens sit at (i, i, i) for their index i,
    picture tokens at their row and column of the picture's grid, and padding goes on from the
    last position.  "clef-flash - Core AI" §Core AI shape: image token k sits at row k // W, column
    k % W, and from the <|vision_end|> index (picture start + N) on the positions move back by
    N - max(H, W).  Reading (the plainest one those numbers allow): image token k at index s + k
    has (s, s + k // W, s + k % W), so the token after the block continues at s + max(H, W), one
    past the largest picture position.
    """
    n = grid_h * grid_w
    pos = np.empty((L, 3), dtype=np.int64)
    for i in range(L):
        if n == 0 or i < image_start:
            pos[i] = (i, i, i)
        elif i < image_start + n:
            k = i - image_start
            pos[i] = (image_start, image_start + k // grid_w, image_start + k % grid_w)
        else:
            p = i - (n - max(grid_h, grid_w))
            pos[i] = (p, p, p)
    return pos


def mrope(x, pos3, rot_dims=ROPE_DIMS, theta=ROPE_THETA):
    """Multimodal rotary: as :func:`rope`, with pair j rotated by pos3[:, plane(j)] * theta^(-2j/64).

    "clef-flash-LiteRT" §Host contract step 5 (cos and sin [L, 64] of the three-plane positions,
    theta = 1e7).  With pos3 = (i, i, i) it is :func:`rope` at position i.
    """
    x = f64(x).copy()
    half = rot_dims // 2
    inv_freq = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / rot_dims)
    pos3 = np.asarray(pos3)
    ang = f64(pos3[:, mrope_planes(rot_dims)]) * inv_freq[None, :]     # [L, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1 = x[..., :half].copy()
    x2 = x[..., half:rot_dims].copy()
    x[..., :half] = x1 * c - x2 * s
    x[..., half:rot_dims] = x2 * c + x1 * s
    return x


def causal_attention(q, k, v):
    """Causal softmax attention with grouped keys/values, one explicit softmax per query row.

    "clef-flash-LiteRT" §Provenance: attention as batched products with an additive mask, the
    grouped keys and values repeated to the query heads.  Query head h reads kv head
    h // (Hq / Hkv); logits are q.k / sqrt(D); row t attends to positions 0..t.
    q: [L, Hq, D]; k, v: [L, Hkv, D].  Returns [L, Hq, D].
    """
    q, k, v = f64(q), f64(k), f64(v)
    L, Hq, D = q.shape
    Hkv = k.shape[1]
    rep = Hq // Hkv
    out = np.empty((L, Hq, D))
    scale = 1.0 / np.sqrt(D)
    mask = np.tril(np.ones((L, L), dtype=bool))
    for h in range(Hq):
        g = h // rep
        logits = (q[:, h, :] @ k[:, g, :].T) * scale          # [L, L]
        logits = np.where(mask, logits, -np.inf)
        m = logits.max(axis=1, keepdims=True)
        p = np.exp(logits - m)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out

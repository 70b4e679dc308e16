"""The chunked (WY) form of the gated delta rule equals the per-token recurrence (CPU, fp64).

The CUDA scan evaluates the recurrence chunk by chunk ("clef-flash-LiteRT" §Provenance: there the
GatedDeltaNet recurrence is exported in 64-position chunks).  This test writes the
chunk algebra out in numpy and checks it against the oracle's token-by-token recurrence for
chunk widths 1, 16 and 64 (width 1 reduces the chunk algebra to the recurrence itself).

Per chunk of C rows with entering state S0 [dv, dk], g = cumulative log(alpha) inside the chunk:
  A[r, s]   = beta_r exp(g_r - g_s) k_r.k_s  (s < r),   T = (I + A)^-1
  W         = T diag(beta exp(g)) K,        U' = T diag(beta) V
  U         = U' - W S0^T
  O         = (diag(exp(g)) Q S0^T + (tril(Q K^T) o exp(g_r - g_s)) U) / sqrt(dk)
  S_C       = exp(g_C) S0 + U^T diag(exp(g_C - g)) K
"""
import numpy as np
import pytest

from oracle import layers as Lr


def chunked_delta_rule(q, k, v, alpha, beta, C):
    L, Hk, dk = k.shape
    Hv, dv = v.shape[1:]
    rep = Hv // Hk
    out = np.zeros((L, Hv, dv))
    S = np.zeros((Hv, dv, dk))
    for h in range(Hv):
        Sh = np.zeros((dv, dk))
        for c0 in range(0, L, C):
            sl = slice(c0, min(L, c0 + C))
            Q, K, V = q[sl, h // rep], k[sl, h // rep], v[sl, h]
            b = beta[sl, h]
            g = np.cumsum(np.log(alpha[sl, h]))
            n = K.shape[0]
            G = np.exp(g[:, None] - g[None, :])
            A = np.tril(b[:, None] * G * (K @ K.T), -1)
            T = np.linalg.inv(np.eye(n) + A)
            W = T @ ((b * np.exp(g))[:, None] * K)
            Up = T @ (b[:, None] * V)
            U = Up - W @ Sh.T
            O = np.exp(g)[:, None] * (Q @ Sh.T) + (np.tril(Q @ K.T) * G) @ U
            out[sl, h] = O / np.sqrt(dk)
            Sh = np.exp(g[-1]) * Sh + U.T @ (np.exp(g[-1] - g)[:, None] * K)
        S[h] = Sh
    return out, S


@pytest.mark.parametrize("C", [1, 16, 64])
def test_chunked_equals_recurrence(C):
    rng = np.random.default_rng(C)
    L, Hk, Hv, d = 150, 2, 4, 32          # ragged last chunk for C = 16, 64
    q = Lr.l2norm(rng.normal(size=(L, Hk, d)))
    k = Lr.l2norm(rng.normal(size=(L, Hk, d)))
    v = rng.normal(size=(L, Hv, d))
    alpha = np.exp(-np.logaddexp(0, rng.normal(size=(L, Hv))) * 0.1)
    beta = 1 / (1 + np.exp(-rng.normal(size=(L, Hv))))
    o_ref, S_ref = Lr.gated_delta_rule(q, k, v, alpha, beta)
    o, S = chunked_delta_rule(q, k, v, alpha, beta, C)
    np.testing.assert_allclose(o, o_ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S, S_ref, rtol=1e-9, atol=1e-11)

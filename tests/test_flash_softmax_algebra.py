"""The flash kernel's online softmax equals the oracle's causal attention (CPU, fp64).

The CUDA attention never forms a full row of logits: for each query row it walks the keys in tiles
of 64 and keeps a reference maximum m_ref, a running sum l and an accumulator.  Scores are turned
into p = 2^((s - m_ref) log2 e) with one fused multiply-add, and m_ref moves (rescaling l and the
accumulator by 2^((m_ref - m_new) log2 e)) only when a tile's maximum exceeds it by more than 8 in
base-2 units, so p stays at most 2^8 and fits the fp16 P operand.  The output is acc / l.  This test
writes that algorithm out in numpy and checks it against the oracle's one-softmax-per-row
definition ("clef-flash-LiteRT" README, "Provenance": grouped keys and values, causal mask), and
that the bound on p holds, including rows whose maximum grows steadily or jumps late.
"""
import numpy as np
import pytest

from oracle import layers as Lr

TILE, RESCALE = 64, 8.0
LOG2E = 1.4426950408889634


def online_attention(q, k, v):
    L, Hq, D = q.shape
    rep = Hq // k.shape[1]
    out = np.empty((L, Hq, D))
    pmax = 0.0
    for h in range(Hq):
        g = h // rep
        for t in range(L):
            m_ref, l, acc = -np.inf, 0.0, np.zeros(D)
            for j0 in range(0, t + 1, TILE):
                keys = np.arange(j0, min(j0 + TILE, t + 1))
                s = k[keys, g, :] @ q[t, h, :] / np.sqrt(D)
                m_new = max(m_ref, s.max())
                if m_ref == -np.inf or (m_new - m_ref) * LOG2E > RESCALE:
                    f = 0.0 if m_ref == -np.inf else 2.0 ** ((m_ref - m_new) * LOG2E)
                    l, acc, m_ref = l * f, acc * f, m_new
                p = 2.0 ** (s * LOG2E - m_ref * LOG2E)
                pmax = max(pmax, p.max())
                l += p.sum()
                acc += p @ v[keys, g, :]
            out[t, h] = acc / l
    return out, pmax


@pytest.mark.parametrize("kind", ["normal", "growing", "late_jump"])
def test_online_softmax_equals_oracle(kind):
    rng = np.random.default_rng(len(kind))
    L, Hq, Hkv, D = 200, 4, 1, 32
    q = rng.standard_normal((L, Hq, D))
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    if kind == "growing":      # logits of later keys keep rising: many small max updates
        k *= (1.0 + np.arange(L) / 20.0)[:, None, None]
    elif kind == "late_jump":  # one key far above the rest late in the row: a large rescale
        k[150] *= 40.0
    got, pmax = online_attention(q, k, v)
    ref = Lr.causal_attention(q, k, v)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-12)
    assert pmax <= 2.0 ** RESCALE * (1 + 1e-12)

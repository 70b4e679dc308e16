"""Causal GQA attention with rotary and output gate (GPU) against the oracle's full softmax."""
import numpy as np
import pytest

import synth
from oracle import layers as Lr
from tests._util import min_row_cosine, rel_rmse

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402

TOL = 5e-3


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def oracle_attn(q, k, v, gate):
    L = q.shape[0]
    pos = np.arange(L)
    o = Lr.causal_attention(Lr.rope(q, pos), Lr.rope(k, pos), v)
    if gate is not None:
        o = o * Lr.sigmoid(gate)
    return o


# L: single position, ragged tiles, a full 64-key tile, the blocked-key lengths 4,032 / 4,096
@pytest.mark.parametrize("B,L,gated", [(1, 1, True), (1, 7, True), (1, 64, False), (2, 97, True),
                                       (1, 300, True), (1, 4032, True), (1, 4096, True)])
def test_attention_matches_oracle(B, L, gated):
    seed = 100 + L
    q = synth.normal_f16(seed, "att.q", 0, (B, L, 16, 256))
    k = synth.normal_f16(seed, "att.k", 0, (B, L, 4, 256))
    v = synth.normal_f16(seed, "att.v", 0, (B, L, 4, 256))
    gate = synth.normal_f16(seed, "att.g", 0, (B, L, 16, 256)) if gated else None
    o = clef.gqa_attn_prefill(_dev(q), _dev(k), _dev(v), None if gate is None else _dev(gate))
    clef.sync_status()
    o = o.double().cpu().numpy()
    for b in range(B):
        ref = oracle_attn(q[b], k[b], v[b], None if gate is None else gate[b])
        assert rel_rmse(o[b], ref) < TOL
        assert min_row_cosine(o[b].reshape(L * 16, 256), ref.reshape(L * 16, 256)) > 0.999


def test_attention_uniform_query_is_prefix_mean():
    # q = 0: every key weighs the same, o_t = mean(v_0..t) (rotary leaves q = 0 at 0)
    L = 130
    q = np.zeros((1, L, 16, 256), np.float16)
    k = synth.normal_f16(1, "att.k", 0, (1, L, 4, 256))
    v = synth.normal_f16(1, "att.v", 0, (1, L, 4, 256))
    o = clef.gqa_attn_prefill(_dev(q), _dev(k), _dev(v)).double().cpu().numpy()[0]
    means = np.cumsum(v[0].astype(np.float64), axis=0) / np.arange(1, L + 1)[:, None, None]
    assert rel_rmse(o, np.repeat(means, 4, axis=1)) < 2e-3


def test_attention_deterministic():
    q = _dev(synth.normal_f16(2, "q", 0, (1, 200, 16, 256)))
    k = _dev(synth.normal_f16(2, "k", 0, (1, 200, 4, 256)))
    v = _dev(synth.normal_f16(2, "v", 0, (1, 200, 4, 256)))
    assert torch.equal(clef.gqa_attn_prefill(q, k, v), clef.gqa_attn_prefill(q, k, v))

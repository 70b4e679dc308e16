"""Chunked prefill with carried state (GPU, clef_prefill_forward_chunk) against the one-shot
prefill and the oracle.

Calls of L1, L2, .. positions on one state must give the rows of a single prefill of the whole
request: the conv history, the recurrent state and the key/value caches carry the earlier
positions.  Both sides compute the same function with different rounding (other chunk and tile
boundaries, fp32 additions in another order), so GPU-vs-GPU the bound is 1e-2 (the scale of two
independently rounded runs), and against the oracle 2e-2 (the final-state bound).
"""
import numpy as np
import pytest

import synth
from oracle import model as om
from tests._util import min_row_cosine, rel_rmse

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402
from full_attention_prefill_gb300.model import PrefillState, synth_model  # noqa: E402

SAME_TOL = 1e-2
FINAL_TOL = 2e-2


@pytest.fixture(scope="module")
def small():
    # 4 layers (3 GDN + 1 attention), a 4,000-row vocabulary prefix of the embedding table
    seed, n_layers, vocab = 3, 4, 4000
    embed = synth.normal_f16(seed, "embed", -1, (vocab, 4096), 0.0, 0.02)
    m = synth_model(seed, n_layers, embed=embed)
    ids = synth.uniform_int(seed, "chunk-ids", -1, (2, 130), vocab)
    whole = m.forward(torch.from_numpy(ids).cuda())
    clef.sync_status()
    return seed, n_layers, m, ids, whole.double().cpu().numpy()


def _chunked(m, ids, sizes, ctx):
    st = PrefillState(m, ids.shape[0], ctx)
    rows, p = [], 0
    for n in sizes:
        out = m.forward_chunk(torch.from_numpy(np.ascontiguousarray(ids[:, p:p + n])).cuda(), st)
        rows.append(out.double().cpu().numpy())
        p += n
        assert st.pos == p
    clef.sync_status()
    return np.concatenate(rows, axis=1)


# chunk lengths: the 64-position calls of the pages' serving mode with a short tail; chunks off
# the 64-position grid (scan chunks and key tiles straddle calls); chunks of 1 and 2 positions
# (the conv history then mixes carried and new rows)
@pytest.mark.parametrize("sizes", [(64, 64, 2), (100, 30), (1, 2, 61, 66)])
def test_chunked_equals_whole(small, sizes):
    seed, n_layers, m, ids, whole = small
    got = _chunked(m, ids, sizes, ctx=192)
    for b in range(2):
        e = rel_rmse(got[b], whole[b])
        print(f"chunks {sizes} b={b}: rel-RMSE vs whole {e:.2e}, "
              f"min row cos {min_row_cosine(got[b], whole[b]):.7f}")
        assert e < SAME_TOL and min_row_cosine(got[b], whole[b]) > 0.9999


def test_chunked_matches_oracle(small):
    seed, n_layers, m, ids, _ = small
    got = _chunked(m, ids, (64, 64, 2), ctx=130)
    ref = om.prefill(ids[1], synth.embedding_rows(seed, ids[1]), lambda l: synth.layer_weights(seed, l),
                     synth.final_norm_weight(seed), n_layers=n_layers)
    e = rel_rmse(got[1], ref)
    print(f"chunks vs oracle: rel-RMSE {e:.2e}")
    assert e < FINAL_TOL


def test_chunk_past_the_state_is_refused(small):
    _, _, m, ids, _ = small
    st = PrefillState(m, 2, 70)
    m.forward_chunk(torch.from_numpy(np.ascontiguousarray(ids[:, :64])).cuda(), st)
    with pytest.raises(clef.ClefError) as e:
        m.forward_chunk(torch.from_numpy(np.ascontiguousarray(ids[:, 64:72])).cuda(), st)
    assert e.value.code == 3          # CLEF_E_TOO_LONG: refused, never cut
    assert st.pos == 64               # a refused call leaves the state where it was
    clef.sync_status()


def test_shared_state_reused_by_two_question_parts(small):
    """Shared-state pair ("clef-flash-LiteRT" card, "Other forms measured"): the shared part is
    prefilled once, then two different question parts each continue their own copy of its state;
    each must equal the one-call prefill of shared part + its questions, and the shared state must
    stay untouched."""
    seed, n_layers, m, ids, whole = small
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    shared = ids[:, :100]
    st = PrefillState(m, 2, 192)
    m.forward_chunk(dev(shared), st)
    before = [t.clone() for t in (st.conv, st.rec, st.kcache, st.vcache)]
    qa = ids[:, 100:130]
    qb = synth.uniform_int(seed, "chunk-ids-b", -1, (2, 45), 4000)
    sa, sb = st.clone(), st.clone()
    out_a = m.forward_chunk(dev(qa), sa).double().cpu().numpy()
    out_b = m.forward_chunk(dev(qb), sb).double().cpu().numpy()
    clef.sync_status()
    assert (st.pos, sa.pos, sb.pos) == (100, 130, 145)
    assert all(torch.equal(a, b) for a, b in zip(before, (st.conv, st.rec, st.kcache, st.vcache)))
    whole_b = m.forward(dev(np.concatenate([shared, qb], axis=1))).double().cpu().numpy()
    clef.sync_status()
    for b in range(2):
        ea = rel_rmse(out_a[b], whole[b, 100:])
        eb = rel_rmse(out_b[b], whole_b[b, 100:])
        print(f"shared state b={b}: questions A vs whole {ea:.2e}, questions B vs whole {eb:.2e}")
        assert ea < SAME_TOL and eb < SAME_TOL
        assert min_row_cosine(out_a[b], whole[b, 100:]) > 0.9999
    assert rel_rmse(out_a[0], out_b[0, :30]) > 0.1      # different questions, different rows

"""The hybrid prefill (GPU, through clef_prefill_forward) against the oracle's prefill."""
import numpy as np
import pytest

import synth
from oracle import model as om
from tests._util import min_row_cosine, rel_rmse

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402
from full_attention_prefill_gb300.model import synth_model  # noqa: E402

FINAL_TOL = 2e-2      # the target's bound on the final hidden states


def oracle_prefill(seed, ids, n_layers):
    return om.prefill(ids, synth.embedding_rows(seed, ids), lambda l: synth.layer_weights(seed, l),
                      synth.final_norm_weight(seed), n_layers=n_layers)


def test_small_model_batch_and_ragged_length():
    # 4 layers (3 GDN + 1 attention), two requests of a ragged length, a 4,000-row vocabulary
    # prefix of the embedding table (same rows as the full table)
    seed, n_layers, B, L, vocab = 3, 4, 2, 130, 4000
    embed = synth.normal_f16(seed, "embed", -1, (vocab, 4096), 0.0, 0.02)
    m = synth_model(seed, n_layers, embed=embed)
    ids = synth.uniform_int(seed, "ids", -1, (B, L), vocab)
    hid = m.forward(torch.from_numpy(ids).cuda())
    clef.sync_status()
    hid = hid.double().cpu().numpy()
    for b in range(B):
        ref = oracle_prefill(seed, ids[b], n_layers)
        e = rel_rmse(hid[b], ref)
        print(f"4-layer b={b}: rel-RMSE {e:.2e}, min row cos {min_row_cosine(hid[b], ref):.6f}")
        assert e < FINAL_TOL


def test_bad_token_is_reported():
    seed, n_layers, vocab = 3, 4, 4000
    embed = synth.normal_f16(seed, "embed", -1, (vocab, 4096), 0.0, 0.02)
    m = synth_model(seed, n_layers, embed=embed)
    ids = torch.full((1, 8), 5, dtype=torch.int32, device="cuda")
    ids[0, 3] = vocab + 7
    m.forward(ids)
    with pytest.raises(clef.ClefError) as e:
        clef.sync_status()
    assert e.value.code == 9


def test_too_long_is_refused():
    seed = 3
    embed = synth.normal_f16(seed, "embed", -1, (16, 4096), 0.0, 0.02)
    m = synth_model(seed, 1, embed=embed)
    ids = torch.zeros((1, 16385), dtype=torch.int32, device="cuda")
    with pytest.raises(clef.ClefError) as e:
        m.forward(ids)
    assert e.value.code == 3


@pytest.mark.slow
def test_full_model_l512():
    """32 layers, L = 512, batch 1, full vocabulary: the decision-request bucket."""
    seed, L = 0, 512
    m = synth_model(seed, 32)
    ids = synth.token_ids(seed, 1, L)
    hid = m.forward(torch.from_numpy(ids).cuda())
    clef.sync_status()
    hid = hid.double().cpu().numpy()[0]
    ref = oracle_prefill(seed, ids[0], 32)
    e = rel_rmse(hid, ref)
    print(f"32-layer L=512: rel-RMSE {e:.2e}, min row cos {min_row_cosine(hid, ref):.6f}")
    assert e < FINAL_TOL


@pytest.mark.slow
def test_reproducible_prefill_is_bit_identical():
    """With CLEF_MODEL_REPRODUCIBLE the split residual adds of a short prefill are summed in part
    order, so two runs of the same 32-layer L = 512 request give the same bits; the result stays
    within fp32 rounding of the default (unordered) path."""
    seed, L = 0, 512
    m = synth_model(seed, 32)
    ids = torch.from_numpy(synth.token_ids(seed, 1, L)).cuda()
    fast = m.forward(ids).clone()
    m.set_reproducible(True)
    try:
        a = m.forward(ids).clone()
        b = m.forward(ids).clone()
        clef.sync_status()
    finally:
        m.set_reproducible(False)
    assert torch.equal(a, b)
    assert rel_rmse(a.double().cpu().numpy(), fast.double().cpu().numpy()) < 1e-2

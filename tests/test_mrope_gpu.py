"""Prefill of requests holding a picture block (GPU, clef_prefill_forward_image) against the
oracle: the picture's rows replace the embedding rows at its tokens and the attention layers
rotate with M-RoPE positions ("clef-flash-LiteRT" README, "Host contract" steps 4-5;
"clef-flash - Core AI" README, "Core AI shape")."""
import numpy as np
import pytest

import synth
from oracle import layers as Lr
from oracle import model as om
from tests._util import min_row_cosine, rel_rmse

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402
from full_attention_prefill_gb300.model import synth_model  # noqa: E402

FINAL_TOL = 2e-2
SEED, N_LAYERS, VOCAB = 3, 4, 4000


@pytest.fixture(scope="module")
def small():
    embed = synth.normal_f16(SEED, "embed", -1, (VOCAB, 4096), 0.0, 0.02)
    return synth_model(SEED, N_LAYERS, embed=embed)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# picture grids: a 4 x 5 block at the pages' index 37, a 1 x 7 strip, a 6 x 2 block starting at 0
@pytest.mark.parametrize("L,start,grid", [(96, 37, (4, 5)), (70, 10, (1, 7)), (40, 0, (6, 2))])
def test_picture_prefill_matches_oracle(small, L, start, grid):
    B, n = 2, grid[0] * grid[1]
    ids = synth.uniform_int(SEED, f"mm-ids-{L}", -1, (B, L), VOCAB)
    rows = synth.normal_f16(SEED, f"image-rows-{L}", -1, (B, n, 4096), 0.0, 0.05)
    hid = small.forward_image(_dev(ids), _dev(rows), start, grid)
    clef.sync_status()
    hid = hid.double().cpu().numpy()
    pos3 = Lr.mrope_positions(L, start, *grid)
    for b in range(B):
        emb = synth.embedding_rows(SEED, ids[b]).astype(np.float64)
        emb[start:start + n] = rows[b]
        run = lambda pos: om.prefill(ids[b], emb, lambda l: synth.layer_weights(SEED, l),  # noqa: E731
                                     synth.final_norm_weight(SEED), n_layers=N_LAYERS, positions=pos)
        ref = run(pos3)
        e = rel_rmse(hid[b], ref)
        print(f"picture {grid} at {start}, L={L}, b={b}: rel-RMSE {e:.2e}, "
              f"min row cos {min_row_cosine(hid[b], ref):.6f}")
        assert e < FINAL_TOL
        if b == 0:
            # the comparison sees the rotary: against the same oracle with plain 1-D positions
            # the GPU rows from the picture on are several times further off
            e1 = rel_rmse(hid[0, start:], run(np.arange(L))[start:])
            em = rel_rmse(hid[0, start:], ref[start:])
            print(f"  rows {start}..: vs M-RoPE oracle {em:.2e}, vs 1-D-position oracle {e1:.2e}")
            assert e1 > 4 * em


# Short prefills split the residual-add GEMMs over K and the parts add in any order, so two runs
# of the same request agree to fp32 rounding, not bit for bit: same-function checks use 1e-3
# (a wrong rotary moves rows by 1e-2 and more).
RERUN_TOL = 1e-3


def test_no_picture_is_the_text_prefill(small):
    ids = synth.uniform_int(SEED, "mm-text", -1, (2, 50), VOCAB)
    a = small.forward(_dev(ids)).double().cpu().numpy()
    b = small.forward_image(_dev(ids), None, 0, (0, 0)).double().cpu().numpy()
    clef.sync_status()
    e = rel_rmse(b, a)
    print(f"no picture vs text prefill: rel-RMSE {e:.2e}")
    assert e < RERUN_TOL


def test_rows_before_the_picture_do_not_see_it(small):
    """Causality: two different pictures (and grids) at index 20 leave rows 0..19 as they are."""
    L, start = 60, 20
    ids = synth.uniform_int(SEED, "mm-grid", -1, (1, L), VOCAB)
    r1 = synth.normal_f16(SEED, "mm-grid-rows", -1, (1, 16, 4096), 0.0, 0.05)
    r2 = synth.normal_f16(SEED, "mm-grid-rows2", -1, (1, 16, 4096), 0.0, 0.05)
    a = small.forward_image(_dev(ids), _dev(r1), start, (4, 4)).double().cpu().numpy()[0]
    b = small.forward_image(_dev(ids), _dev(r2), start, (2, 8)).double().cpu().numpy()[0]
    clef.sync_status()
    before, after = rel_rmse(a[:start], b[:start]), rel_rmse(a[start:], b[start:])
    print(f"two pictures: rows before {before:.2e}, rows from the picture on {after:.2e}")
    assert before < RERUN_TOL and after > 0.1


def test_bad_picture_arguments(small):
    ids = _dev(synth.uniform_int(SEED, "mm-bad", -1, (1, 30), VOCAB))
    rows = torch.zeros((1, 12, 4096), dtype=torch.float16, device="cuda")
    with pytest.raises(clef.ClefError) as e:
        small.forward_image(ids, rows, 25, (3, 4))          # does not fit in 30 tokens
    assert e.value.code == 2
    with pytest.raises(clef.ClefError) as e:
        small.forward_image(ids, rows, -1, (3, 4))
    assert e.value.code == 1

"""The benchmark's full-size prefills against rows the oracle computed (GPU).

The stored rows (tests/golden/, written by tests/golden/make_prefill_goldens.py, which calls only
the synthetic-input module and the oracle) are final-norm hidden rows of
  * one request of 16,384 positions through all 32 layers (prefill_l16384_rows.npz), and
  * requests 0, 13 and 31 of the 32 requests of 512 positions (prefill_b32x512_rows.npz),
with the benchmark's weights (seed 0) and token ids (seed 1000).  The GPU side runs exactly the
benchmark's launch configuration (clef_prefill_forward on all requests at once).  Each stored row
must be within the 32-layer bound of 2e-2 relative RMSE, element by element over the row.
"""
import os

import numpy as np
import pytest

import synth
from tests._util import min_row_cosine, rel_rmse

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402
from full_attention_prefill_gb300.model import synth_model  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FINAL_TOL = 2e-2


@pytest.fixture(scope="module")
def model():
    return synth_model(0, 32)


def _check_rows(got, ref, what):
    errs = [rel_rmse(got[i], ref[i]) for i in range(len(ref))]
    cos = min_row_cosine(got, ref)
    print(f"{what}: {len(ref)} rows, worst row rel-RMSE {max(errs):.2e}, all rows "
          f"{rel_rmse(got, ref):.2e}, min row cosine {cos:.6f}")
    assert max(errs) < FINAL_TOL
    return errs


def test_l16384_against_oracle_rows(model):
    g = np.load(os.path.join(GOLDEN, "prefill_l16384_rows.npz"))
    assert int(g["weight_seed"]) == 0
    ids = synth.token_ids(int(g["ids_seed"]), 1, 16384)
    out = model.forward(torch.from_numpy(ids).cuda())
    clef.sync_status()
    pos = torch.from_numpy(g["positions"]).cuda()
    got = out[0, pos].double().cpu().numpy()
    _check_rows(got, g["rows"].astype(np.float64), "32 layers, L=16384")


def test_b32x512_against_oracle_rows(model):
    g = np.load(os.path.join(GOLDEN, "prefill_b32x512_rows.npz"))
    assert int(g["weight_seed"]) == 0
    ids = synth.token_ids(int(g["ids_seed"]), 32, 512)
    out = model.forward(torch.from_numpy(ids).cuda())
    clef.sync_status()
    pos = torch.from_numpy(g["positions"]).cuda()
    for i, r in enumerate(g["requests"]):
        got = out[int(r), pos].double().cpu().numpy()
        _check_rows(got, g["rows"][i].astype(np.float64), f"32 x 512, request {int(r)}")

"""Non-finite hidden rows are reported, not returned as an answer (GPU).

"Clef-Flash-ANE-LUT6", section "Vision weights": the largest residual met (about 12,400) is within
FP16's range, and inputs that overflow FP16 are rejected rather than answered.  Here an inf is
written into the embedding row of one token of a request (an ordinary input, not a fault): the
prefill must report CLEF_E_NONFINITE through the status word, naming a row no later than that
token; clef_check_finite must flag that row and every later row of the request (by causality
the inf reaches all of them), and rows of earlier chunks must stay finite and unflagged.  A
clean request reports nothing.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402
from full_attention_prefill_gb300.model import synth_model  # noqa: E402


@pytest.fixture(scope="module")
def model():
    return synth_model(0, 4)


def test_clean_request_reports_nothing(model):
    ids = torch.from_numpy(synth.token_ids(31, 1, 130)).cuda()
    out = model.forward(ids)
    clef.sync_status()
    flags = clef.check_finite(out)
    clef.sync_status()
    assert int(flags.sum()) == 0


@pytest.mark.parametrize("pos", [0, 57, 129])
def test_inf_in_an_embedding_row_is_reported(model, pos):
    L = 130
    ids_np = synth.token_ids(32, 2, L)
    tok = int(ids_np[1, pos])
    # other occurrences of the same token id would also carry the inf; make pos the first one
    assert not np.any(ids_np[1, :pos] == tok) and not np.any(ids_np[0] == tok)
    ids = torch.from_numpy(ids_np).cuda()
    saved = model.embed[tok].clone()
    try:
        model.embed[tok, 7] = float("inf")
        out = model.forward(ids)
        with pytest.raises(clef.ClefError) as e:
            clef.sync_status()
        assert e.value.code == 7                               # CLEF_E_NONFINITE
        msg = clef.lib().clef_last_error().decode()
        first = int(msg.split("hidden row ")[1].split()[0])
        chunk0 = (pos // 64) * 64
        assert L + chunk0 <= first <= L + pos                  # request 1, not before pos's chunk
        clef.sync_status()                                     # the report was cleared
        flags = clef.check_finite(out).cpu().numpy().reshape(2, L)
        with pytest.raises(clef.ClefError):
            clef.sync_status()
        assert flags[0].sum() == 0                             # the other request is untouched
        assert flags[1, pos:].all()                            # pos and every later row
        assert not flags[1, :chunk0].any()                     # earlier chunks stay finite
        assert torch.isfinite(out[1, :chunk0].float()).all()
    finally:
        model.embed[tok] = saved
    out = model.forward(ids)
    clef.sync_status()


def test_check_finite_flags_rows_of_any_array():
    x = torch.zeros((5, 24), dtype=torch.float16, device="cuda")
    x[1, 3] = float("nan")
    x[4, 23] = float("-inf")
    flags = clef.check_finite(x)
    with pytest.raises(clef.ClefError) as e:
        clef.sync_status()
    assert e.value.code == 7 and "hidden row 1 " in clef.lib().clef_last_error().decode()
    assert flags.cpu().tolist() == [0, 1, 0, 0, 1]

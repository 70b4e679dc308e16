"""The joint schema head (GPU, through clef_joint_head) against the oracle's head.

Bounds: the GPU runs fp16 activations between its kernels (fp32 accumulation and an fp32
residual stream across six layers), so logits agree to 1e-2 relative RMSE and probabilities to
5e-3 absolute; per-question sums are 1 to fp32 rounding and a one-option question gives 1.
"""
import numpy as np
import pytest

import synth
from oracle import head as ohead
from tests._util import rel_rmse

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402
from full_attention_prefill_gb300.head import DeviceHead  # noqa: E402

LOGIT_TOL, PROB_TOL = 1e-2, 5e-3


@pytest.fixture(scope="module")
def weights():
    return synth.head_weights(0)


@pytest.fixture(scope="module")
def dhead(weights):
    return DeviceHead(weights)


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=dtype)).cuda()


def _gpu(dhead, hidden, r):
    return dhead(_dev(hidden, np.float16), _dev(r["q_avg"], np.float32), _dev(r["o_avg"], np.float32),
                 _dev(r["g_avg"], np.float32), _dev(r["lexical"], np.float32), _dev(r["member"], np.uint8),
                 _dev(r["type_ids"], np.int32), _dev(r["q_valid"], np.uint8), _dev(r["o_valid"], np.uint8),
                 _dev(r["key_valid"], np.uint8))


# (T, option counts per question): a small request, a ragged one with invalid entries, the
# pages' largest padded shape (16 questions, 128 options) over 4,096 rows, and a long request
CASES = [(200, [2, 3, 1, 4], False), (517, [3, 2, 5, 1], True), (4096, [8] * 16, False),
         (16384, [2, 4, 3], False)]


@pytest.mark.parametrize("T,questions,holes", CASES)
def test_head_matches_oracle(dhead, weights, T, questions, holes):
    hidden = synth.normal_f16(T, "head.hidden", 0, (T, 4096))
    r = synth.head_request(T + 1, T, questions)
    if holes:
        r["q_valid"][1] = 0
        r["o_valid"][0] = 0
        r["key_valid"][-7:] = 0
    lg, p = _gpu(dhead, hidden, r)
    clef.sync_status()
    lg, p = lg.double().cpu().numpy(), p.double().cpu().numpy()
    ref_lg, ref_p = ohead.joint_head(hidden.astype(np.float64), weights, r["q_avg"], r["o_avg"], r["g_avg"],
                                     r["lexical"], r["member"], r["type_ids"], r["q_valid"], r["o_valid"],
                                     r["key_valid"])
    e = rel_rmse(lg, ref_lg)
    dp = np.abs(p - ref_p).max()
    print(f"head T={T} Q={len(questions)} O={sum(questions)}: logits rel-RMSE {e:.2e}, max |dp| {dp:.2e}")
    assert e < LOGIT_TOL and dp < PROB_TOL
    for q in range(len(questions)):
        sel = r["member"][q].astype(bool) & r["o_valid"].astype(bool)
        if r["q_valid"][q] and sel.any():
            assert abs(p[sel].sum() - 1.0) < 1e-5
        else:
            assert np.all(p[sel] == 0)
    if 1 in questions and not holes:
        o = int(np.cumsum([0] + questions)[questions.index(1)])
        assert p[o] == 1.0


def test_head_refuses_too_many_options(dhead):
    hidden = torch.zeros((64, 4096), dtype=torch.float16, device="cuda")
    r = synth.head_request(1, 64, [1])
    big = np.zeros((129, 64))
    with pytest.raises(clef.ClefError) as e:
        dhead(hidden, _dev(r["q_avg"], np.float32), _dev(big, np.float32), _dev(r["g_avg"], np.float32),
              _dev(np.zeros((129, 4096)), np.float32), _dev(np.zeros((1, 129)), np.uint8),
              _dev(r["type_ids"], np.int32))
    assert e.value.code == 2

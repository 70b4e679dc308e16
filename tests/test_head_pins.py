"""Pins of the joint schema head's oracle (CPU only).

"clef-flash - Core AI" README, Readout contract: each question's probabilities are a softmax over
that question's options; the head averages the hidden rows over each span, reads the last token
as a global vector and averages the lm_head rows of each option's ids.  The layers between are a
reading (oracle/csrc/head.cpp); these tests check what holds for any weights of that form, and
the C++ oracle against its independent numpy twin.
"""
import numpy as np

import synth
from oracle import head
from oracle.twin import head as thead

T = 96
W = synth.head_weights(0)
HID = synth.normal_f16(0, "head.hidden", 0, (T, 4096)).astype(np.float64)


def _run(r, hidden=HID, w=W, **kw):
    args = dict(q_avg=r["q_avg"], o_avg=r["o_avg"], g_avg=r["g_avg"], lexical=r["lexical"],
                member=r["member"], type_ids=r["type_ids"], q_valid=r["q_valid"],
                o_valid=r["o_valid"], key_valid=r["key_valid"])
    args.update(kw)
    return head.joint_head(hidden, w, **args)


def test_probabilities_sum_to_one_per_question_and_single_option_is_certain():
    r = synth.head_request(1, T, [2, 3, 1, 4])
    _, p = _run(r)
    for q in range(4):
        assert abs(p[r["member"][q].astype(bool)].sum() - 1.0) < 1e-12
    assert p[5] == 1.0                                   # question 2 has one option (index 5)
    assert np.all(p > 0) and np.all(p <= 1)


def test_matches_numpy_twin():
    r = synth.head_request(2, T, [3, 2, 5])
    r["q_valid"][1] = 0                                  # one question left out
    r["o_valid"][4] = 0                                  # one option left out
    r["key_valid"][-10:] = 0                             # padding rows
    lg, p = _run(r)
    tl, tp = thead.joint_head(HID, W, r["q_avg"], r["o_avg"], r["g_avg"], r["lexical"], r["member"],
                              r["type_ids"], r["q_valid"], r["o_valid"], r["key_valid"])
    assert np.abs(lg - tl).max() < 1e-11 * np.abs(tl).max()
    assert np.abs(p - tp).max() < 1e-12
    assert p[3] == 0 and p[4] == 0                       # question 1's options, option 4


def test_options_are_permutation_equivariant():
    """Reordering the options of a question (their spans, lexical rows and member columns)
    reorders the logits and probabilities the same way."""
    r = synth.head_request(3, T, [4, 2])
    lg, p = _run(r)
    perm = np.array([2, 0, 3, 1, 4, 5])
    lg2, p2 = _run(r, o_avg=r["o_avg"][perm], lexical=r["lexical"][perm], member=r["member"][:, perm],
                   o_valid=r["o_valid"][perm])
    np.testing.assert_allclose(lg2, lg[perm], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(p2, p[perm], rtol=1e-11, atol=1e-13)


def test_identical_options_get_equal_probability():
    r = synth.head_request(4, T, [3])
    r["o_avg"][2] = r["o_avg"][0]
    r["lexical"][2] = r["lexical"][0]
    _, p = _run(r)
    assert abs(p[0] - p[2]) < 1e-14 and abs(p.sum() - 1.0) < 1e-12


def test_padding_rows_do_not_matter():
    """Rows outside every span, flagged invalid as keys, and not the last token, do not change
    the result."""
    r = synth.head_request(5, T, [2, 2])
    r["key_valid"][70:90] = 0
    lg, _ = _run(r)
    other = HID.copy()
    other[70:90] = synth.normal_f64(9, "head.noise", 0, (20, 4096))
    lg2, _ = _run(r, hidden=other)
    np.testing.assert_allclose(lg2, lg, rtol=1e-12, atol=1e-14)
    # while a valid key row outside every span does change it (the layers read every token)
    r["key_valid"][70:90] = 1
    lg3, _ = _run(r)
    lg4, _ = _run(r, hidden=other)
    assert np.abs(lg3 - lg4).max() > 1e-6


def test_span_means_and_global_row_are_what_the_layers_read():
    """The head sees a span only through its mean: replacing a question's span rows by their mean
    (repeated) leaves the result unchanged when those rows are invisible as keys."""
    r = synth.head_request(6, T, [2, 1])
    a, b = r["q_span"][0]
    r["key_valid"][a:b] = 0
    lg, _ = _run(r)
    flat = HID.copy()
    flat[a:b] = HID[a:b].mean(axis=0)
    lg2, _ = _run(r, hidden=flat)
    np.testing.assert_allclose(lg2, lg, rtol=1e-10, atol=1e-12)

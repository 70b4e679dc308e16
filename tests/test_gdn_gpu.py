"""The chunked gated-delta-rule scan (GPU) against the oracle's per-token recurrence."""
import numpy as np
import pytest

import synth
from oracle import layers as Lr
from tests._util import min_row_cosine, rel_rmse

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402

# Per-layer budget of the target is 5e-3 relative RMSE; the scan alone is held to the same bound.
TOL = 5e-3


def scan_inputs(seed, B, L):
    """Smoke-config inputs: q, k N(0,1) L2-normalised, v N(0,1) (all fp16);
    beta = sigmoid(N(0,1)), alpha = exp(-softplus(N(0,1)) * 0.1) (fp32)."""
    q = synth.normal_f64(seed, "gdn.q", 0, (B, L, 16, 128))
    k = synth.normal_f64(seed, "gdn.k", 0, (B, L, 16, 128))
    q = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(np.float16)
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float16)
    v = synth.normal_f16(seed, "gdn.v", 0, (B, L, 32, 128))
    na = synth.normal_f64(seed, "gdn.na", 0, (B, L, 32))
    nb = synth.normal_f64(seed, "gdn.nb", 0, (B, L, 32))
    alpha = np.exp(-np.logaddexp(0.0, na) * 0.1).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-nb))).astype(np.float32)
    return q, k, v, alpha, beta


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gpu(q, k, v, alpha, beta, s0=None, want_state=False):
    r = clef.gdn_prefill(_dev(q), _dev(k), _dev(v), _dev(alpha), _dev(beta),
                         None if s0 is None else _dev(s0), want_state=want_state)
    clef.sync_status()
    return r


@pytest.mark.parametrize("B,L", [(1, 128), (1, 1), (1, 63), (1, 65), (2, 150), (1, 1024)])
def test_scan_matches_recurrence(B, L):
    q, k, v, alpha, beta = scan_inputs(B * 1000 + L, B, L)
    o, S = run_gpu(q, k, v, alpha, beta, want_state=True)
    o = o.double().cpu().numpy()
    S = S.double().cpu().numpy()
    for b in range(B):
        o_ref, S_ref = Lr.gated_delta_rule(q[b], k[b], v[b], alpha[b], beta[b])
        err = rel_rmse(o[b], o_ref)
        assert err < TOL, (b, err)
        assert min_row_cosine(o[b].reshape(L, -1), o_ref.reshape(L, -1)) > 0.999
        assert rel_rmse(S[b], S_ref) < TOL


def test_scan_with_initial_state():
    B, L = 1, 100
    q, k, v, alpha, beta = scan_inputs(7, B, L)
    s0 = synth.normal_f32(7, "gdn.s0", 0, (B, 32, 128, 128), 0.0, 0.3)
    o, S = run_gpu(q, k, v, alpha, beta, s0=s0, want_state=True)
    o_ref, S_ref = Lr.gated_delta_rule(q[0], k[0], v[0], alpha[0], beta[0], s0[0])
    assert rel_rmse(o.double().cpu().numpy()[0], o_ref) < TOL
    assert rel_rmse(S.double().cpu().numpy()[0], S_ref) < TOL


def test_scan_invariant_beta0_alpha1():
    # beta = 0, alpha = 1: the state never changes and o_t = S0 q_t / sqrt(128)
    B, L = 1, 70
    q, k, v, _, _ = scan_inputs(11, B, L)
    s0 = synth.normal_f32(11, "gdn.s0", 0, (B, 32, 128, 128), 0.0, 0.3)
    alpha = np.ones((B, L, 32), np.float32)
    beta = np.zeros((B, L, 32), np.float32)
    o, S = run_gpu(q, k, v, alpha, beta, s0=s0, want_state=True)
    np.testing.assert_allclose(S.cpu().numpy(), s0, rtol=0, atol=0)
    ref = np.einsum("hij,thj->thi", s0[0].astype(np.float64),
                    np.repeat(q[0], 2, axis=1).astype(np.float64)) / np.sqrt(128)
    assert rel_rmse(o.double().cpu().numpy()[0], ref) < 2e-3


def test_scan_invariant_alpha0_beta1():
    # alpha = 0, beta = 1: S_t = v_t k_t^T (the state is replaced at every step)
    B, L = 1, 66
    q, k, v, _, _ = scan_inputs(12, B, L)
    alpha = np.zeros((B, L, 32), np.float32)
    beta = np.ones((B, L, 32), np.float32)
    o, S = run_gpu(q, k, v, alpha, beta, want_state=True)
    ref = np.einsum("hi,hj->hij", v[0, -1].astype(np.float64),
                    np.repeat(k[0, -1], 2, axis=0).astype(np.float64))
    assert rel_rmse(S.double().cpu().numpy()[0], ref) < 2e-3


def test_scan_alpha1_beta1_maps_k_to_v():
    # alpha = 1, beta = 1, unit k: after step t the state maps k_t to v_t
    B, L = 1, 64
    q, k, v, _, _ = scan_inputs(13, B, L)
    alpha = np.ones((B, L, 32), np.float32)
    beta = np.ones((B, L, 32), np.float32)
    _, S = run_gpu(q, k, v, alpha, beta, want_state=True)
    kt = np.repeat(k[0, -1], 2, axis=0).astype(np.float64)
    kt /= np.linalg.norm(kt, axis=-1, keepdims=True)
    got = np.einsum("hij,hj->hi", S.double().cpu().numpy()[0], kt)
    assert rel_rmse(got, v[0, -1]) < 5e-3


def test_scan_deterministic():
    q, k, v, alpha, beta = scan_inputs(5, 1, 300)
    a = run_gpu(q, k, v, alpha, beta)
    b = run_gpu(q, k, v, alpha, beta)
    assert torch.equal(a, b)


# A scan of one request with at least 64 chunks runs in pieces (the chunk phase of the next
# piece overlapping the state pass of this one, on two streams); three requests run in one pass.  The state crosses pieces in fp32, exactly as it stays in tensor memory in one pass, so the
# same request must come out bit for bit the same either way, with or without an entering state.
@pytest.mark.parametrize("L,with_s0", [(4096, False), (8192, True), (4150, True)])
def test_pieces_equal_one_pass(L, with_s0):
    q, k, v, alpha, beta = scan_inputs(L + int(with_s0), 1, L)
    s0 = synth.normal_f32(L, "gdn.s0p", 0, (1, 32, 128, 128), 0.0, 0.3) if with_s0 else None
    rep = lambda a: np.concatenate([a, a, a], axis=0)  # noqa: E731
    o1, S1 = run_gpu(q, k, v, alpha, beta, s0=s0, want_state=True)
    o3, S3 = run_gpu(rep(q), rep(k), rep(v), rep(alpha), rep(beta),
                     s0=None if s0 is None else rep(s0), want_state=True)
    assert torch.equal(o1[0], o3[0]) and torch.equal(o1[0], o3[2])
    assert torch.equal(S1[0], S3[0])
    # without a state output the pieces carry the state through the workspace's scratch
    o0 = run_gpu(q, k, v, alpha, beta, s0=s0, want_state=False)
    assert torch.equal(o0[0], o1[0])
    # and against the recurrence on the first 256 positions (their own prefix)
    o_ref, _ = Lr.gated_delta_rule(q[0, :256], k[0, :256], v[0, :256], alpha[0, :256], beta[0, :256],
                                   s0=None if s0 is None else s0[0])
    assert rel_rmse(o1[0, :256].double().cpu().numpy(), o_ref) < TOL

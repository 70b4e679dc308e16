"""The prefill's kernels at the benchmark's full size (16,384 positions), in the launch
configuration the benchmark times, checked on sampled outputs that the fp64 oracle computes one by
one (GPU).

* LUT-6 GEMM: the prefill's five weight shapes at M = 16,384 tokens; 384 sampled outputs each,
  against fp64 dot products of the token row with the dequantised weight row.
* Attention: 16,384 positions, 6 sampled query positions (the first, the last, and rows across the
  key tiles) x all 16 heads, against the oracle's causal attention (one explicit softmax per row)
  computed for those rows only, after the oracle's rotary.
* Gated delta rule: 16,384 positions (a long single request: the scan runs in pieces on two
  streams), value heads 0, 1 (key head 0) and 14, 15 (key head 7), outputs and final state,
  against the oracle's per-token recurrence restricted to those heads.
"""
import numpy as np
import pytest

import synth
from oracle import layers as Lr
from oracle import lut6 as olut
from tests._util import rel_rmse

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402

M = 16384


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# (N, K) of the fused GDN input projection, the attention input projection, the output
# projections, the interleaved gate/up projection and the down projection
@pytest.mark.parametrize("N,K", [(12288, 4096), (10240, 4096), (4096, 4096), (24576, 4096),
                                 (4096, 12288)])
def test_gemm_full_size_sampled(N, K):
    x = synth.normal_f16(0, "fs.x", K, (M, K))
    packed, lut = synth.lut6_weight(0, "fs.w", N + K, N, K)
    y = clef.lut6_gemm(_dev(x), _dev(packed), _dev(lut))
    clef.sync_status()
    rng = np.random.default_rng(N + K)
    ms = rng.integers(0, M, 384)
    ns = rng.integers(0, N, 384)
    ms[:2], ns[:2] = (0, M - 1), (0, N - 1)                   # the corners
    got = y[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()].double().cpu().numpy()
    ref = np.empty(384)
    for i, (m, n) in enumerate(zip(ms, ns)):
        g = n // 16
        w = olut.dequant(packed[16 * g:16 * g + 16], lut[g:g + 1], 16, K)[n - 16 * g]
        ref[i] = x[m].astype(np.float64) @ w
    e = rel_rmse(got, ref)
    print(f"GEMM {M} x {N} x {K}: sampled rel-RMSE {e:.2e}")
    assert e < 1e-3


def test_attention_full_size_sampled():
    q = synth.normal_f16(0, "q", 0, (1, M, 16, 256))
    k = synth.normal_f16(0, "k", 0, (1, M, 4, 256))
    v = synth.normal_f16(0, "v", 0, (1, M, 4, 256))
    o = clef.gqa_attn_prefill(_dev(q), _dev(k), _dev(v))
    clef.sync_status()
    rows = [0, 63, 64, 5000, 12345, M - 1]
    got = o[0, rows].double().cpu().numpy()
    pos = np.arange(M)
    kr = Lr.rope(k[0], pos)
    qr = Lr.rope(q[0, rows], np.array(rows))
    qfull = np.zeros((M, 16, 256))
    qfull[rows] = qr
    vv = v[0].astype(np.float64)
    # the oracle's causal attention, computing only the sampled query rows
    ref = np.concatenate([Lr.causal_attention(qfull, kr, vv, rows=(t, t + 1)) for t in rows])
    e = rel_rmse(got, ref)
    print(f"attention L={M}: sampled rows rel-RMSE {e:.2e}")
    assert e < 5e-3


def test_gdn_full_size_sampled_heads():
    q = synth.normal_f64(1, "gdn.q", 0, (1, M, 16, 128))
    k = synth.normal_f64(1, "gdn.k", 0, (1, M, 16, 128))
    q = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(np.float16)
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float16)
    v = synth.normal_f16(1, "gdn.v", 0, (1, M, 32, 128))
    na = synth.normal_f64(1, "gdn.na", 0, (1, M, 32))
    nb = synth.normal_f64(1, "gdn.nb", 0, (1, M, 32))
    alpha = np.exp(-np.logaddexp(0.0, na) * 0.1).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-nb))).astype(np.float32)
    o, S = clef.gdn_prefill(_dev(q), _dev(k), _dev(v), _dev(alpha), _dev(beta), want_state=True)
    clef.sync_status()
    o = o[0].double().cpu().numpy()
    S = S[0].double().cpu().numpy()
    for kh in (0, 7):
        hv = [2 * kh, 2 * kh + 1]
        o_ref, S_ref = Lr.gated_delta_rule(q[0][:, [kh]], k[0][:, [kh]], v[0][:, hv],
                                           alpha[0][:, hv], beta[0][:, hv])
        e = rel_rmse(o[:, hv], o_ref)
        es = rel_rmse(S[hv], S_ref)
        print(f"GDN L={M}: value heads {hv}: out rel-RMSE {e:.2e}, final state {es:.2e}")
        assert e < 5e-3 and es < 5e-3

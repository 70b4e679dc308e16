"""LUT-6 kernels against the oracle (GPU): bit-exact dequant, then the tcgen05 GEMM."""
import numpy as np
import pytest

import synth
from oracle import lut6 as olut
from tests._util import rel_rmse

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("n,k", [(4096, 4096), (48, 12), (16, 64), (12288, 4096)])
def test_dequant_bit_exact(n, k):
    packed, lut = synth.lut6_weight(0, "dq", 0, n, k)
    w = clef.lut6_dequant(_dev(packed), _dev(lut), k).cpu().numpy()
    ref = olut.dequant_f16(packed, lut, n, k)
    assert np.array_equal(w.view(np.uint16), ref.view(np.uint16))


# (m, n, k): config-0 smoke size, ragged m, ragged n (not a multiple of the 128-row tile),
# one k-block, several k-blocks with a ring wrap, a tall m spanning many tiles, and two tall
# cases spanning more CTAs than the GPU has SMs (persistent walk: several tiles per CTA)
CASES = [(128, 4096, 4096), (77, 256, 128), (300, 784, 320), (1, 16, 64), (129, 512, 64 * 7),
         (1000, 1024, 1024), (4100, 1296, 128), (2600, 2048, 64 * 3),
         # the prefill's projection shapes at a short and a middle length
         (512, 12288, 4096), (512, 4096, 12288), (4096, 4096, 4096),
         # 384-token tiles (launches whose wide tiles fill the GPU): ragged m, a partial last
         # channel tile with a 3-step k (the accumulators drained after 2 steps of the next
         # tile), a 1-step k, and several tiles per CTA
         (4100, 4608, 1024), (2600, 4624, 64 * 3), (3000, 6144, 64), (6000, 8192, 512)]


@pytest.mark.parametrize("m,n,k", CASES)
@pytest.mark.parametrize("fp32", [False, True])
def test_gemm_matches_oracle(m, n, k, fp32):
    x = synth.normal_f16(0, "x", m, (m, k))
    packed, lut = synth.lut6_weight(0, "w", n + k, n, k)
    y = clef.lut6_gemm(_dev(x), _dev(packed), _dev(lut), out_fp32=fp32)
    clef.sync_status()
    y = y.double().cpu().numpy()
    ref = olut.linear(x, packed, lut, n)
    rms = np.sqrt(np.mean(ref ** 2))
    if fp32:
        # fp16 x fp16 products are exact; the tensor core's fp32 accumulation over k terms loses
        # about 2^-23 * sqrt(k) * rms (7.6e-6 rms at k = 4096): bound it at 1e-4 rms
        np.testing.assert_allclose(y, ref, rtol=1e-3, atol=1e-4 * rms)
        assert rel_rmse(y, ref) < 2e-5
    else:
        # plus one rounding to fp16 (unit roundoff 2^-11)
        np.testing.assert_allclose(y, ref, rtol=1e-3, atol=1e-3 * rms)
        assert rel_rmse(y, ref) < 1e-3


def test_gemm_empty_m_is_noop():
    packed, lut = synth.lut6_weight(0, "w", 1, 256, 64)
    x = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    y = clef.lut6_gemm(x, _dev(packed), _dev(lut))
    assert y.shape == (0, 256)


def test_gemm_rejects_bad_shapes():
    packed, lut = synth.lut6_weight(0, "w", 1, 256, 64)
    x = torch.zeros((4, 60), dtype=torch.float16, device="cuda")
    with pytest.raises(clef.ClefError) as e:
        clef.lut6_gemm(x, _dev(packed), _dev(lut))
    assert e.value.code == 2


@pytest.mark.parametrize("m,n", [(512, 1024), (4096, 8192)])
def test_gemm_deterministic(m, n):
    x = _dev(synth.normal_f16(3, "x", 0, (m, 1024)))
    packed, lut = synth.lut6_weight(3, "w", 0, n, 1024)
    p, l = _dev(packed), _dev(lut)
    a = clef.lut6_gemm(x, p, l)
    b = clef.lut6_gemm(x, p, l)
    assert torch.equal(a, b)


def test_tile_layout_moves_whole_quadruples():
    # the tiled layout documented in clef.h, restated with numpy index arithmetic
    n, k = 48, 192
    packed = synth.random_bytes(5, "tile", 0, (n, k * 3 // 4))
    tiled = clef.lut6_tile(_dev(packed), k).cpu().numpy().reshape(-1)
    trip = packed.reshape(n, k // 4, 3)
    expect = np.empty((n // 16, k // 64, 32, 2, 4, 3), dtype=np.uint8)
    for G in range(n // 16):
        for kb in range(k // 64):
            for t in range(32):
                for h in range(2):
                    for j in range(4):
                        expect[G, kb, t, h, j] = trip[16 * G + t // 4 + 8 * h, 16 * kb + 4 * j + t % 4]
    assert np.array_equal(tiled, expect.reshape(-1))


def test_canonical_entry_equals_tiled_entry():
    """clef_lut6_gemm_canonical on the card's own packing gives the same bits as clef_lut6_gemm on
    the tiled permutation, and refuses a workspace smaller than its size query."""
    import ctypes
    m, n, k = 300, 784, 320
    x = _dev(synth.normal_f16(4, "x", 0, (m, k)))
    packed, lut = synth.lut6_weight(4, "w", 0, n, k)
    p, l = _dev(packed), _dev(lut)
    a = clef.lut6_gemm(x, p, l)                                  # canonical bytes in
    b = clef.lut6_gemm(x, clef.lut6_tile(p, k), l, tiled=True)   # tiled once, then multiplied
    clef.sync_status()
    assert torch.equal(a, b)
    need = clef.lib().clef_lut6_gemm_canonical_workspace_size(n, k)
    assert need == n * k * 3 // 4
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    y = torch.empty((m, n), dtype=torch.float16, device="cuda")
    rc = clef.lib().clef_lut6_gemm_canonical(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(p.data_ptr()), ctypes.c_void_p(l.data_ptr()),
        ctypes.c_void_p(y.data_ptr()), 0, m, n, k, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 8                                               # CLEF_E_WORKSPACE

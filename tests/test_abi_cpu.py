"""The C-ABI library loads on a machine without a GPU and exports every declared symbol; its
host-side LUT-6 packing agrees with the oracle's.  No compute call touches a device here."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import lut6 as olut

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    hdr = open(os.path.join(ROOT, "include", "clef.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(clef_[a-z0-9_]+)\s*\(", hdr)))


@pytest.fixture(scope="module")
def lib():
    import full_attention_prefill_gb300 as clef
    if not os.path.exists(clef.LIB_PATH):
        from full_attention_prefill_gb300 import _build
        _build.build()
    return clef.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "clef_lut6_gemm" in names and "clef_prefill_forward" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_host_pack_matches_oracle(lib):
    import full_attention_prefill_gb300 as clef
    rng = np.random.default_rng(0)
    idx = rng.integers(0, 64, size=(37, 96), dtype=np.uint8)
    assert np.array_equal(clef.lut6_pack(idx), olut.pack(idx))
    assert np.array_equal(clef.lut6_unpack(olut.pack(idx), 96), idx)


def test_host_pack_rejects_bad_input(lib):
    import full_attention_prefill_gb300 as clef
    with pytest.raises(clef.ClefError) as e:
        clef.lut6_pack(np.full((2, 8), 64, dtype=np.uint8))
    assert e.value.code == 1
    with pytest.raises(clef.ClefError) as e:
        clef.lut6_pack(np.zeros((2, 6), dtype=np.uint8))
    assert e.value.code == 2


def test_version(lib):
    assert lib.clef_version() >> 16 == 1 and lib.clef_version() & 0xFFFF >= 1


def test_gate_up_interleave_layout():
    from full_attention_prefill_gb300 import SWIGLU_BLOCK
    from full_attention_prefill_gb300.model import interleave_gate_up
    b = SWIGLU_BLOCK
    n = 4 * b
    gp = np.arange(n * 3, dtype=np.int64).reshape(n, 3).astype(np.uint8)
    up = (gp.astype(np.int64) + 101).astype(np.uint8)
    gl = np.arange(n // 16 * 64, dtype=np.float32).reshape(n // 16, 64).astype(np.float16)
    ul = gl + np.float16(1000)
    p, l = interleave_gate_up((gp, gl), (up, ul))
    for j in range(n // b):
        assert np.array_equal(p[2 * j * b:(2 * j + 1) * b], gp[j * b:(j + 1) * b])
        assert np.array_equal(p[(2 * j + 1) * b:(2 * j + 2) * b], up[j * b:(j + 1) * b])
        t = b // 16
        assert np.array_equal(l[2 * j * t:(2 * j + 1) * t], gl[j * t:(j + 1) * t])
        assert np.array_equal(l[(2 * j + 1) * t:(2 * j + 2) * t], ul[j * t:(j + 1) * t])


@pytest.mark.parametrize("L,s,h,w", [(46, 37, 2, 3), (50, 0, 0, 0), (300, 37, 14, 14),
                                     (120, 37, 8, 8), (20, 3, 1, 7), (64, 0, 8, 8)])
def test_host_mrope_positions_match_oracle(lib, L, s, h, w):
    import full_attention_prefill_gb300 as clef
    from oracle import layers as Lr
    assert np.array_equal(clef.mrope_positions(L, s, (h, w)), Lr.mrope_positions(L, s, h, w))


def test_host_mrope_positions_errors(lib):
    import full_attention_prefill_gb300 as clef
    with pytest.raises(clef.ClefError) as e:
        clef.mrope_positions(40, 37, (2, 3))          # the picture does not fit
    assert e.value.code == 2
    with pytest.raises(clef.ClefError) as e:
        clef.mrope_positions(40, 0, (2, 0))           # half a grid
    assert e.value.code == 1


@pytest.mark.parametrize("B", [1, 2, 3, 32])
@pytest.mark.parametrize("L", [1, 64, 1024, 4095, 4096, 4150, 8192, 16384])
def test_gdn_workspace_regions_fit(lib, B, L):
    """The scan's workspace carving stays inside the size it reports and no regions overlap, for
    every shape class (one pass, pieces with the carried-state scratch, with and without the
    gated norm's o).  A mismatch of the two once let a pieced scan write past its workspace."""
    nch, M = -(-L // 64), B * L
    sizes = [M * 32 * 4,                      # g
             B * nch * 32 * 64 * 4,           # exp(g)
             B * nch * 64 * 32 * 128 * 2,     # W
             B * nch * 64 * 32 * 128 * 4,     # U'
             B * nch * 64 * 32 * 128 * 2,     # decayed keys
             B * nch * 32 * 64 * 64 * 2,      # Aqk^T
             B * 32 * 128 * 128 * 4,          # carried state
             M * 32 * 128 * 2]                # o
    for with_norm in (0, 1):
        offs = (ctypes.c_int64 * 8)()
        total = ctypes.c_int64()
        assert lib.clef_debug_gdn_workspace_layout(B, L, with_norm, offs, ctypes.byref(total)) == 0
        regions = sorted((o, sz) for o, sz in zip(offs, sizes) if o >= 0)
        for o, sz in regions:
            assert 0 <= o and o + sz <= total.value, (B, L, with_norm, o, sz, total.value)
        for (a, sa), (b, _) in zip(regions, regions[1:]):
            assert a + sa <= b
        assert (offs[6] >= 0) == (B == 1 and nch >= 64)     # the scan runs in pieces
        assert (offs[7] >= 0) == bool(with_norm)


def test_binding_fails_loudly_without_the_library(tmp_path):
    """The product path has no fallback: with the library's file absent the binding raises."""
    import subprocess
    import sys
    code = (
        "import full_attention_prefill_gb300 as clef\n"
        f"clef.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
        "clef._lib = None\n"
        "try:\n"
        "    clef.lib()\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "else:\n"
        "    print('no error')\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT,
                       timeout=300)
    assert "raised:" in r.stdout and "no fallback" in r.stdout, r.stdout + r.stderr

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
    assert lib.clef_version() >> 16 == 1

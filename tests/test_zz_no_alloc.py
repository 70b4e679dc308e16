"""The allocation-free GDN scan (clef_gdn_prefill_noalloc) against the workspace version.

Some callers cannot allocate device memory themselves (a plugin inside a runtime that owns the
allocator, or a serving loop that must not allocate), so the library offers a scan whose scratch
is a fixed array inside the library.  This test calls it through the C ABI twice in a row, with
different inputs, and checks each result against clef_gdn_prefill on the same inputs: both run the
same kernels in the same order, so outputs and final states must be equal bit for bit, and the
second call must not see anything the first one left in the shared scratch.  One call enters
from a given state and one returns no state.  Sizes beyond the built-in scratch, and batch sizes
whose token count is out of range, are refused.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

from tests.test_gdn_gpu import scan_inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402
import synth  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def noalloc(q, k, v, alpha, beta, s0=None, want_state=True):
    B, L = q.shape[0], q.shape[1]
    o = torch.empty((B, L, 32, 128), dtype=torch.float16, device="cuda")
    s_out = torch.empty((B, 32, 128, 128), dtype=torch.float32, device="cuda") if want_state else None
    rc = clef.lib().clef_gdn_prefill_noalloc(_p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(s0), _p(o),
                                             _p(s_out), B, L, _stream())
    assert rc == 0, clef.lib().clef_last_error()
    clef.sync_status()
    return o, s_out


def test_noalloc_matches_workspace_scan_twice():
    cases = (
        (21, 1, 1000, False, True),    # one request, no entering state, state returned
        (22, 2, 150, True, True),      # two requests entering from a given state
        (23, 1, 333, False, False),    # no state returned
    )
    for seed, B, L, with_s0, want_state in cases:
        q, k, v, alpha, beta = (_dev(a) for a in scan_inputs(seed, B, L))
        s0 = _dev(synth.normal_f32(seed, "noalloc.s0", 0, (B, 32, 128, 128), 0.0, 0.1)) if with_s0 else None
        o, s = noalloc(q, k, v, alpha, beta, s0, want_state)
        o_ref, s_ref = clef.gdn_prefill(q, k, v, alpha, beta, s0=s0, want_state=True)
        clef.sync_status()
        assert torch.equal(o, o_ref), f"outputs differ (seed {seed})"
        if want_state:
            assert torch.equal(s, s_ref), f"final states differ (seed {seed})"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    B, L = 1, 4096
    q = torch.zeros((B, L, 16, 128), dtype=torch.float16, device="cuda")
    v = torch.zeros((B, L, 32, 128), dtype=torch.float16, device="cuda")
    a = torch.ones((B, L, 32), dtype=torch.float32, device="cuda")
    o = torch.empty_like(v)
    rc = clef.lib().clef_gdn_prefill_noalloc(_p(q), _p(q), _p(v), _p(a), _p(a), None, _p(o), None, B, L,
                                             _stream())
    assert rc == 2
    assert b"scratch" in clef.lib().clef_last_error()
    # a batch whose token count is beyond 2^22 is refused before any size product is formed
    # (the pointers are never read: validation comes first)
    for huge_b in (1 << 57, 1 << 62):
        rc = clef.lib().clef_gdn_prefill_noalloc(_p(q), _p(q), _p(v), _p(a), _p(a), None, _p(o), None,
                                                 huge_b, 1, _stream())
        assert rc == 2, clef.lib().clef_last_error()
        assert b"4194304" in clef.lib().clef_last_error()

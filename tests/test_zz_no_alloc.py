"""The allocation-free GDN scan (clef_gdn_prefill_noalloc) against the workspace version.

Some callers cannot allocate device memory themselves (a plugin inside a runtime that owns the
allocator, or a serving loop that must not allocate), so the library offers a scan whose scratch
is a fixed array inside the library.  This test calls it through the C ABI twice in a row, with
different inputs, and checks each result against clef_gdn_prefill on the same inputs: the second
call must not see anything the first one left in the shared scratch.  It also checks that a size
beyond the built-in scratch is refused.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

from tests._util import rel_rmse
from tests.test_gdn_gpu import TOL, scan_inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import full_attention_prefill_gb300 as clef  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def noalloc(q, k, v, alpha, beta):
    B, L = q.shape[0], q.shape[1]
    o = torch.empty((B, L, 32, 128), dtype=torch.float16, device="cuda")
    s_out = torch.empty((B, 32, 128, 128), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = clef.lib().clef_gdn_prefill_noalloc(_p(q), _p(k), _p(v), _p(alpha), _p(beta), None, _p(o),
                                             _p(s_out), B, L, stream)
    assert rc == 0, clef.lib().clef_last_error()
    clef.sync_status()
    return o, s_out


def test_noalloc_matches_workspace_scan_twice():
    for seed, (B, L) in ((21, (1, 1000)), (22, (2, 150))):
        q, k, v, alpha, beta = (_dev(a) for a in scan_inputs(seed, B, L))
        o, s = noalloc(q, k, v, alpha, beta)
        o_ref, s_ref = clef.gdn_prefill(q, k, v, alpha, beta, want_state=True)
        clef.sync_status()
        assert rel_rmse(o.double().cpu().numpy(), o_ref.double().cpu().numpy()) < TOL
        assert rel_rmse(s.double().cpu().numpy(), s_ref.double().cpu().numpy()) < TOL


def test_noalloc_refuses_sizes_beyond_its_scratch():
    B, L = 1, 4096
    q = torch.zeros((B, L, 16, 128), dtype=torch.float16, device="cuda")
    v = torch.zeros((B, L, 32, 128), dtype=torch.float16, device="cuda")
    a = torch.ones((B, L, 32), dtype=torch.float32, device="cuda")
    o = torch.empty_like(v)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = clef.lib().clef_gdn_prefill_noalloc(_p(q), _p(q), _p(v), _p(a), _p(a), None, _p(o), None, B, L,
                                             stream)
    assert rc == 2
    assert b"scratch" in clef.lib().clef_last_error()

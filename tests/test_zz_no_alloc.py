"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Plugins run by an engine that owns every device allocation, and serving loops whose memory
pool is fixed at start-up, have no way to hand this library a workspace.  This entry point
keeps its routing scratch in a static device array inside the library instead.  The test
calls it through the C ABI twice in a row (the array keeps the first call's contents) and
checks both results against moe_debug_route, the workspace-based entry point, and against the
CPU oracle's routing: integers bit-exact, routing weights within the 1e-6 relative tolerance of
the routing parity tests.

This file is named to be collected last, so that a run stopping at the first failure has
already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import nvfp4_expert_gemms_gb300 as M
import synth

pytestmark = pytest.mark.gpu

MAX_TOKENS = 2048  # MOE_ROUTE_NOALLOC_MAX_TOKENS in include/moe_gb300.h


def _noalloc(logits, k):
    lib = M.lib()
    f = lib.moe_route_noalloc
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int] + [C.c_void_p] * 6
    T, E = (int(s) for s in logits.shape)
    dev = logits.device
    idx = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    w = torch.full((T, k), -1.0, dtype=torch.float32, device=dev)
    off = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((T * k,), -1, dtype=torch.int32, device=dev)
    inv = torch.full((T * k,), -1, dtype=torch.int32, device=dev)
    st = f(logits.data_ptr(), T, E, k, idx.data_ptr(), w.data_ptr(), off.data_ptr(), perm.data_ptr(),
           inv.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st, (idx, w, off, perm, inv)


def _with_workspace(logits, k):
    T, E = (int(s) for s in logits.shape)
    d = M.moe_packed_size("fp8", E, 128, 128)
    ws = torch.empty(M.moe_workspace_size(d, T, k), dtype=torch.uint8, device=logits.device)
    return M.moe_debug_route(logits, k, ws)


def _same(a, b):
    for i, (x, y) in enumerate(zip(a, b)):
        if i == 1:
            np.testing.assert_allclose(x.cpu().numpy(), y.cpu().numpy(), rtol=1e-6, atol=0)
        else:
            assert torch.equal(x, y), i


def test_noalloc_route_matches_workspace_route_twice(orc):
    cases = [(2048, 128, 8, 1.1), (37, 16, 4, None)]  # the maximum size, then a small ragged one
    for n, (T, E, k, zipf) in enumerate(cases):
        lg = synth.gen_logits(T, E, seed=100 + n, zipf_alpha=zipf)
        logits = torch.from_numpy(lg).cuda()
        st, got = _noalloc(logits, k)
        assert st == 0, M.moe_status_string(st)
        want = _with_workspace(logits, k)
        torch.cuda.synchronize()
        _same(got, want)
        # and against the CPU oracle's routing and permutation
        ridx, rw = orc.route(lg, k)
        roff, rperm, rinv = orc.permute(ridx, E)
        idx, w, off, perm, inv = (t.cpu().numpy() for t in got)
        assert np.array_equal(idx, ridx) and np.array_equal(off, roff)
        assert np.array_equal(perm, rperm) and np.array_equal(inv, rinv)
        np.testing.assert_allclose(w, rw, rtol=1e-6, atol=0)


def test_noalloc_route_rejects_too_many_tokens():
    logits = torch.zeros((MAX_TOKENS + 1, 8), dtype=torch.float32, device="cuda")
    st, _ = _noalloc(logits, 2)
    assert st == 3 and M.moe_status_string(st) == "workspace too small"

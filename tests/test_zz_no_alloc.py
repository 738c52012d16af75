"""GPU: the allocation-free backward (rmsnorm_bwd_noalloc) against the
workspace path.

The allocation-free call is for callers that cannot allocate device memory
where they run the backward (graph capture without a memory pool, serving
loops that forbid allocation, plugins whose host framework owns all device
memory).  It must give the same dx and dweight as rmsnorm_dweight_begin +
rmsnorm_bwd_dx + dweight_finalize with a caller workspace, on two calls in a
row (the second one must not see anything the first left in the shared
scratch), and it must refuse sizes beyond its fixed scratch.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import invariant_rmsnorm_fwd_gb300 as rb

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _case(hidden, lengths, seed, heads=1):
    wl = synth.Workload("na", hidden, np.asarray(lengths), seed=seed)
    n_rows = wl.n_tokens * heads
    x = synth.logical_tensor(wl, synth.TAG_X, n_rows, 1.0, device="cuda").reshape(wl.n_tokens, heads, hidden)
    dy = synth.logical_tensor(wl, synth.TAG_DY, n_rows, 1e-2, device="cuda").reshape(wl.n_tokens, heads, hidden)
    w = synth.weight(wl, device="cuda")
    perm = synth.seeded_permutation(seed, wl.n_tokens).astype(np.int32)   # one permuted call
    idx = torch.as_tensor(perm, device="cuda").long()
    return wl, x[idx].contiguous(), dy[idx].contiguous(), w, perm


def _with_workspace(wl, xp, dp, w, tok, heads):
    cl = rb.call_layout(tok, heads, wl.n_tokens)
    ws = rb.DweightWorkspace(wl.n_tokens * heads, wl.hidden)
    ws.begin()
    dx = rb.rmsnorm_bwd_dx(xp, w, dp, cl, wl.eps, workspace=ws)
    dw = ws.finalize()
    assert ws.status() == 0
    return dx, dw


@pytest.mark.parametrize("hidden,lengths,heads", [(4096, [300, 47, 210], 1), (128, [500, 333], 8)])
def test_noalloc_matches_workspace_path_twice(hidden, lengths, heads):
    for seed in (21, 22):                                   # two calls in a row, different data
        wl, xp, dp, w, tok = _case(hidden, lengths, seed, heads)
        want_dx, want_dw = _with_workspace(wl, xp, dp, w, tok, heads)
        cl = rb.call_layout(tok, heads, wl.n_tokens)
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        dx = torch.full_like(dp, float("nan"))
        _, dw = rb.rmsnorm_bwd_noalloc(xp, w, dp, cl, wl.eps, dx=dx, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(dx.view(torch.int16), want_dx.view(torch.int16))
        assert torch.equal(dw.view(torch.int32), want_dw.view(torch.int32))


def test_noalloc_refuses_sizes_beyond_its_scratch():
    H = 4096
    n = rb.NOALLOC_SCRATCH_BYTES // (H * 4) + 64            # spill area alone exceeds the scratch
    lib = rb._load()
    assert lib.rmsnorm_dweight_workspace_bytes(n, H) > rb.NOALLOC_SCRATCH_BYTES
    cl = rb.call_layout(np.arange(4, dtype=np.int32), 1, n, with_plan=False)
    x = torch.zeros(4, H, dtype=torch.bfloat16, device="cuda")
    dw = torch.zeros(H, device="cuda")
    L = cl.struct(H)
    rc = lib.rmsnorm_bwd_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                                 ctypes.c_void_p(x.data_ptr()), H, 1e-6, ctypes.byref(L), None,
                                 ctypes.c_void_p(dw.data_ptr()), None,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -6                                          # RMSNORM_ERR_WORKSPACE, nothing enqueued


def test_noalloc_without_dx_or_status_and_an_empty_call_reports_missing():
    hidden, lengths = 4096, [300, 47]
    wl, xp, dp, w, tok = _case(hidden, lengths, 31)
    want_dx, want_dw = _with_workspace(wl, xp, dp, w, tok, 1)
    cl = rb.call_layout(tok, 1, wl.n_tokens)
    _, dw = rb.rmsnorm_bwd_noalloc(xp, w, dp, cl, wl.eps)            # no dx, no status
    torch.cuda.synchronize()
    assert torch.equal(dw.view(torch.int32), want_dw.view(torch.int32))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dx = torch.full_like(dp, float("nan"))
    _, dw = rb.rmsnorm_bwd_noalloc(xp, w, dp, cl, wl.eps, dx=dx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(dx.view(torch.int16), want_dx.view(torch.int16))
    assert torch.equal(dw.view(torch.int32), want_dw.view(torch.int32))
    # a call holding none of the multiset's rows, right after a full one: the
    # scratch still holds the previous call's rows, and only the status word
    # can tell that this call's rows never arrived
    empty = rb.call_layout(np.zeros(0, dtype=np.int32), 1, wl.n_tokens)
    status.fill_(-1)
    rb.rmsnorm_bwd_noalloc(xp, w, dp, empty, wl.eps, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & rb.STATUS_MISSING

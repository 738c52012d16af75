"""GPU: the bounded-wait timeout path of the pipelined row kernel.

Every wait of the warp-specialised pipeline gives up after a fixed time,
sets RMSNORM_STATUS_TIMEOUT in the workspace and lets the kernel return, so
that a lost arrival is reported instead of hanging the GPU (issue #270,
"Acceptance criteria": a failure is reported, never hidden by a fallback).

The test needs a wait that nothing completes.  A separate, test-only build of
the library (never the product library) is compiled with
RBI_TEST_WITHHOLD_EMPTY, so the column warps never release a pipeline stage,
and with a 10 ms wait limit.  What then happens, read from the kernel:
 * the first S batches run normally (their stages need no release);
 * the producer's wait to reuse stage 0 runs out before it issues any copy
   into that stage; it raises the CTA's abort flag, sets the status bit, waits
   (bounded) for the copies it issued to the S stages already in use, which
   nothing blocks, and leaves;
 * the stats and column warps wait for a stage the producer never fills;
   each of those waits also runs out after 10 ms and they leave;
 * one CTA per team (hidden 4096), so no cluster barrier is involved.
So the launch ends by itself within a few wait limits.  The test checks the
status bit, that the context is still usable, and that a normal call right
after it, through the product library, gives the same bits as before.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import synth
import invariant_rmsnorm_fwd_gb300 as rb
from invariant_rmsnorm_fwd_gb300 import _build

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _variant():
    path = _build.build_test_variant("waitlimit", {"RBI_TEST_WITHHOLD_EMPTY": None,
                                                   "RBI_WAIT_LIMIT_NS": "10000000ull"})
    lib = ctypes.CDLL(path)
    P, I64, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
    lib.rmsnorm_dweight_begin.argtypes = [P, ctypes.c_size_t, I64, I64, P]
    lib.rmsnorm_bwd_dx.argtypes = [P, P, P, I64, F, ctypes.POINTER(rb._Layout), P, P, P]
    lib.rmsnorm_dweight_begin.restype = lib.rmsnorm_bwd_dx.restype = ctypes.c_int
    return lib


def _product_run(x, w, dy, cl, eps):
    ws = rb.DweightWorkspace(cl.n_logical_tokens, x.shape[1])
    ws.begin()
    dx = rb.rmsnorm_bwd_dx(x, w, dy, cl, eps, workspace=ws)
    dw = ws.finalize()
    return dx, dw, ws.status()


def test_lost_stage_release_times_out_and_reports():
    H, n = 4096, 3000
    wl = synth.Workload("timeout", H, np.array([n]), seed=5)
    x = synth.logical_tensor(wl, synth.TAG_X, n, 1.0, device="cuda")
    dy = synth.logical_tensor(wl, synth.TAG_DY, n, 1e-2, device="cuda")
    w = synth.weight(wl, device="cuda")
    cl = rb.call_layout(np.arange(n, dtype=np.int32), 1, n)
    dx0, dw0, st0 = _product_run(x, w, dy, cl, wl.eps)
    assert st0 == 0

    lib = _variant()
    ws = rb.DweightWorkspace(n, H)
    dx = torch.zeros_like(dy)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    L = cl.struct(H)
    assert lib.rmsnorm_dweight_begin(ctypes.c_void_p(ws.buf.data_ptr()), ws.bytes, n, H, stream) == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.rmsnorm_bwd_dx(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                            ctypes.c_void_p(dy.data_ptr()), H, wl.eps, ctypes.byref(L),
                            ctypes.c_void_p(dx.data_ptr()), ctypes.c_void_p(ws.buf.data_ptr()), stream)
    assert rc == 0
    torch.cuda.synchronize()                              # the launch ends by itself
    elapsed = time.perf_counter() - t0
    status = ws.status()
    assert status & rb.STATUS_TIMEOUT, status
    assert elapsed < 5.0, elapsed

    # the context is still usable and a normal call gives the same bits as before
    dx1, dw1, st1 = _product_run(x, w, dy, cl, wl.eps)
    assert st1 == 0
    assert torch.equal(dx1.view(torch.int16), dx0.view(torch.int16))
    assert torch.equal(dw1.view(torch.int32), dw0.view(torch.int32))

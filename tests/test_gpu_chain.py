"""GPU: residual add fused with the norm, and the loss seed's scale.

* h = bf16(x + r) must equal the oracle's rounding of the exact sum bit for
  bit, and y must equal the plain forward of h bit for bit (fusing changes
  nothing) and match the oracle within the y tolerance.
* dh = bf16(s * dx_norm + dres) within the dx tolerance (cancellation scale
  s*K + |dres|), dweight = s * tree within the dweight tolerance; with s = 1
  and no dres the call is exactly rmsnorm_bwd_dx; the scaled dweight is the
  unscaled one times s in one FP32 multiplication.
* Every layout gives the same bits when every call uses the multiset's
  active-token denominator; a per-call denominator is caught as red.
"""
import numpy as np
import pytest
import torch

import gpu_common as G
import synth
import tolerances as tol
from oracle import chain
from invariant_rmsnorm_fwd_gb300 import harness
from invariant_rmsnorm_fwd_gb300 import layout as L
import invariant_rmsnorm_fwd_gb300 as rb

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _inputs(wl, rpt=1, head_set=0):
    x, dy, w = G.logical_inputs(wl, head_set, rpt)
    n = wl.n_tokens * rpt
    r = synth.logical_tensor(wl, synth.TAG_RES, n, wl.x_std, head_set, device="cuda").reshape(x.shape)
    dres = synth.logical_tensor(wl, synth.TAG_DRES, n, wl.dy_std, head_set, device="cuda").reshape(x.shape)
    return x, r, dy, dres, w


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_chain(run, x, r, dy, dres, w, eps, s, rows=None):
    H = w.shape[0]
    n = x.reshape(-1, H).shape[0]
    rows = G.sample_rows(n) if rows is None else rows
    ridx = torch.as_tensor(rows, device="cuda")
    xs, rs = x.reshape(-1, H)[ridx], r.reshape(-1, H)[ridx]
    h_ref, y_ref, _ = chain.add_forward(xs, rs, w, eps)
    assert np.array_equal(_bits(run.h.reshape(-1, H)[ridx]), h_ref)              # bit exact
    y = run.y.reshape(-1, H)[ridx].float().cpu().numpy()
    rep = [tol.check("y", y, y_ref, tol.bound_y(y_ref))]
    hs = run.h.reshape(-1, H)[ridx]
    dh_ref, k, _, _ = chain.add_backward(hs, w, dy.reshape(-1, H)[ridx], dres.reshape(-1, H)[ridx], eps, s)
    dh = run.dx.reshape(-1, H)[ridx].float().cpu().numpy()
    rep.append(tol.check("dh", dh, dh_ref, tol.bound_dx(dh_ref, k)))
    _, _, dw_ref, sc = chain.add_backward(run.h.reshape(-1, H), w, dy.reshape(-1, H), None, eps, s, want_dx=False)
    rep.append(tol.check("dweight", run.dweight.cpu().numpy(), dw_ref, tol.bound_dw(dw_ref, sc)))
    return rep


@pytest.mark.parametrize("hidden", [8, 64, 128, 256, 264, 1024, 4096, 5120, 8192, 10240, 16384])
def test_chain_matches_oracle_and_is_layout_invariant(hidden):
    wl = synth.Workload("t", hidden, np.asarray([70, 3, 130, 1, 64, 9]), seed=hidden, chunk_rows=37)
    x, r, dy, dres, w = _inputs(wl)
    s = 1.0 / wl.n_tokens                                   # mean over the multiset's active tokens
    lays = L.workload_layouts(wl)
    runs = {k: harness.run_layout_chain(v, x, r, dy, dres, w, wl.eps, s) for k, v in lays.items()}
    rep = harness.assert_batch_invariant(runs, lays)
    assert rep.green, rep.summary()
    assert all(v.status == 0 and v.untouched_padding for v in runs.values())
    for res in _check_chain(runs["full"], x, r, dy, dres, w, wl.eps, s):
        assert res["violations"] == 0, res


def test_fused_forward_equals_add_then_norm():
    wl = synth.config("c1")
    x, r, _, _, w = _inputs(wl)
    H = wl.hidden
    cl = rb.call_layout(np.arange(wl.n_tokens, dtype=np.int32), 1, wl.n_tokens, with_plan=False)
    xp, rp = x.reshape(-1, H), r.reshape(-1, H)
    h, y = rb.rmsnorm_add_fwd(xp, rp, w, cl, wl.eps)
    assert torch.equal(h.view(torch.int16), (xp.float() + rp.float()).to(torch.bfloat16).view(torch.int16))
    y2 = rb.rmsnorm_fwd(h, w, cl, wl.eps)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    # in place over the residual stream: h written into r
    r2 = rp.clone()
    rb.rmsnorm_add_fwd(xp, r2, w, cl, wl.eps, h=r2, y=torch.empty_like(xp))
    assert torch.equal(r2.view(torch.int16), h.view(torch.int16))


@pytest.mark.parametrize("hidden", [128, 4096])
def test_unscaled_without_dres_is_the_plain_backward(hidden):
    wl = synth.Workload("t", hidden, np.asarray([100, 77]), seed=3, chunk_rows=37)
    x, _, dy, _, w = _inputs(wl)
    H = hidden
    cl = rb.call_layout(np.arange(177, dtype=np.int32), 1, 177)
    xp, dp = x.reshape(-1, H), dy.reshape(-1, H)
    ws1 = rb.DweightWorkspace(177, H); ws1.begin()
    dx1 = rb.rmsnorm_bwd_dx(xp, w, dp, cl, wl.eps, workspace=ws1)
    ws2 = rb.DweightWorkspace(177, H); ws2.begin()
    dx2 = rb.rmsnorm_add_bwd(xp, w, dp, cl, wl.eps, workspace=ws2)
    assert torch.equal(dx1.view(torch.int16), dx2.view(torch.int16))
    dw1, dw2 = ws1.finalize(), ws2.finalize(grad_scale=1.0)
    assert torch.equal(dw1.view(torch.int32), dw2.view(torch.int32))
    # the scaled root is the unscaled root times s, one FP32 multiplication
    s = np.float32(1.0 / 177)
    dws = ws2.finalize(grad_scale=float(s)).cpu().numpy()
    assert np.array_equal(dws.view(np.uint32), (dw1.cpu().numpy() * s).astype(np.float32).view(np.uint32))
    # the same with the sharded combine
    roots = torch.stack([ws2.finalize_range(0, 2), ws2.finalize_range(2, 2)])
    dwc = rb.dweight_combine(roots, grad_scale=float(s)).cpu().numpy()
    assert np.array_equal(dwc.view(np.uint32), dws.view(np.uint32))


def test_per_call_denominator_is_caught():
    """The failure the pages name: a loss mean taken over each call's own active
    tokens instead of the multiset's.  The harness must judge it red."""
    wl = synth.config("c0")
    x, r, dy, dres, w = _inputs(wl)
    lays = L.workload_layouts(wl)
    runs = {k: harness.run_layout_chain(v, x, r, dy, dres, w, wl.eps, lambda tok: 1.0 / max(1, int((tok >= 0).sum())))
            for k, v in lays.items()}
    rep = harness.assert_batch_invariant(runs, lays)
    assert not rep.green
    assert any(d.tensor == "dx" and not d.equal for d in rep.diffs)
    good = {k: harness.run_layout_chain(v, x, r, dy, dres, w, wl.eps, 1.0 / wl.n_tokens) for k, v in lays.items()}
    assert harness.assert_batch_invariant(good, lays).green


def test_qk_heads_chain():
    wl = synth.config("c3")
    R = wl.heads[1]
    x, r, dy, dres, w = _inputs(wl, rpt=R, head_set=1)
    s = 1.0 / wl.n_tokens
    lays = L.workload_layouts(wl, ["full", "chunked", "permuted"])
    runs = {k: harness.run_layout_chain(v, x, r, dy, dres, w, wl.eps, s, rows_per_token=R) for k, v in lays.items()}
    rep = harness.assert_batch_invariant(runs, lays)
    assert rep.green, rep.summary()
    for res in _check_chain(runs["full"], x, r, dy, dres, w, wl.eps, s):
        assert res["violations"] == 0, res


def test_bad_scale_is_refused():
    H = 128
    cl = rb.call_layout(np.arange(4, dtype=np.int32), 1, 4, with_plan=False)
    x = torch.zeros(4, H, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    for bad in (float("nan"), float("inf")):
        with pytest.raises(rb.RmsNormError) as e:
            rb.rmsnorm_add_bwd(x, w, x, cl, 1e-6, grad_scale=bad)
        assert e.value.code == -13
    with pytest.raises(rb.RmsNormError):
        rb.rmsnorm_add_fwd(x, x, w, cl, 1e-6, h=x, y=x)           # h and y may not alias

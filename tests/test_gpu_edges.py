"""GPU: exact reduction order, hidden-size sweep, degenerate layouts, status word."""
import numpy as np
import pytest
import torch

import gpu_common as G
import oracle
import synth
from oracle import tree_replay
from invariant_rmsnorm_fwd_gb300 import harness
from invariant_rmsnorm_fwd_gb300 import layout as L
import invariant_rmsnorm_fwd_gb300 as rb

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = "cuda"


def bf16(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(DEV)


def _workload(lengths, hidden, seed=7, x_std=1.0, dy_std=1e-2):
    return synth.Workload("t", hidden, np.asarray(lengths), seed=seed, x_std=x_std, dy_std=dy_std,
                          chunk_rows=37)


# ------------------------------------------------------------------ exact order

@pytest.mark.parametrize("hidden", [8, 128, 4096, 5120])
@pytest.mark.parametrize("n_rows", [1, 63, 64, 65, 259, 4999, 10500])
def test_dweight_follows_the_fixed_tree_bitwise(hidden, n_rows):
    """eps = 0 and rows of constant magnitude 2^k make xhat = +-1 exactly, so the
    leaves are +-dy exactly; dy is chosen so that every association order gives
    different FP32 bits.  The GPU must equal the FP32 replay of the tree.
    10500 rows: 660 quarter units on 152 teams leave 52 in the last round, which
    the backward splits into 8-row eighths (the halves meet in the finalize)."""
    rng = np.random.default_rng(hidden * 1000 + n_rows)
    signs = rng.choice([-1.0, 1.0], size=(n_rows, hidden))
    mags = 2.0 ** rng.integers(-3, 4, size=(n_rows, 1))
    x = signs * mags
    pool = np.array([16777216.0, 1.0, -1.0, 3.0, -16777216.0, 0.5, 2.0 ** -20, 65536.0, -0.0, 255.0])
    dy = pool[rng.integers(0, pool.size, size=(n_rows, hidden))]
    leaves = (dy * signs).astype(np.float32)               # dy * xhat, exact
    want = tree_replay.dweight(leaves)
    lengths = [n_rows]
    for kind in ("full", "chunked", "singleton"):
        lay = L.make_layout(kind, lengths, chunk=37)
        run = harness.run_layout(lay, bf16(x), bf16(dy), bf16(np.ones(hidden)), 0.0)
        assert run.status == 0
        got = run.dweight.cpu().numpy()
        assert got.tobytes() == want.tobytes(), (kind, np.flatnonzero(got != want)[:5])


def test_constant_rows_map_to_w_times_sign_bitwise():
    H = 4096
    wl = _workload([5, 3], H)
    w = synth.weight(wl, device=DEV)
    c = np.array([0.125, -0.5, 3.0, -96.0, 1.0, 0.25, -2.0, 7.5])
    x = np.repeat(c[:, None], H, axis=1)
    lay = L.make_layout("chunked", [8], chunk=3)
    run = harness.run_layout(lay, bf16(x), bf16(np.ones((8, H))), w, 1e-6)
    want = (w.float().cpu()[None, :] * torch.as_tensor(np.sign(c), dtype=torch.float32)[:, None]).to(torch.bfloat16)
    assert torch.equal(run.y.reshape(8, H).cpu().view(torch.int16), want.view(torch.int16))


# ------------------------------------------------------------------ hidden sizes

@pytest.mark.parametrize("hidden", [8, 16, 24, 64, 128, 136, 256, 264, 512, 1024, 4096, 4104, 5120, 6144, 8192,
                                    12288, 16384])
def test_hidden_sweep_invariance_and_accuracy(hidden):
    wl = _workload([70, 3, 130, 1, 64, 9], hidden, seed=hidden)
    x, dy, w, lays, runs = G.run_all_layouts(wl)
    rep = harness.assert_batch_invariant(runs, lays)
    assert rep.green, rep.summary()
    for name in ("full", "singleton"):
        for r in G.oracle_check(runs[name], x, dy, w, wl.eps):
            assert r["violations"] == 0, (name, r)
    assert all(r.untouched_padding for r in runs.values())


# ------------------------------------------------------------------ degenerate layouts

def test_empty_and_all_padding_calls():
    H = 128
    wl = _workload([5, 60], H)
    x, dy, w = G.logical_inputs(wl)
    calls = [np.zeros(0, np.int32), np.full(9, -1, np.int32),
             np.arange(0, 40, dtype=np.int32), np.full(3, -1, np.int32), np.arange(40, 65, dtype=np.int32)]
    lay = L.Layout("odd", calls, 65)
    run = harness.run_layout(lay, x, dy, w, wl.eps)
    ref = harness.run_layout(L.make_layout("full", [65]), x, dy, w, wl.eps)
    for t in ("y", "dx", "dweight"):
        assert harness.bitwise_diff(t, getattr(run, t), getattr(ref, t), "odd", "full").equal
    assert run.status == 0 and run.untouched_padding


def test_empty_multiset_gives_zero_dweight():
    ws = rb.DweightWorkspace(0, 64, device=DEV)
    ws.begin()
    dw = ws.finalize()
    assert torch.equal(dw.cpu(), torch.zeros(64)) and ws.status() == 0


# ------------------------------------------------------------------ paths agree

def test_contrib_only_and_dx_only_match_fused():
    H = 4096
    wl = _workload([100, 50], H)
    x, dy, w = G.logical_inputs(wl)
    cl = rb.call_layout(np.arange(150, dtype=np.int32), 1, 150)
    xp, dp = x.reshape(150, H), dy.reshape(150, H)
    ws1 = rb.DweightWorkspace(150, H); ws1.begin()
    dx1 = rb.rmsnorm_bwd_dx(xp, w, dp, cl, 1e-6, workspace=ws1)
    dw1 = ws1.finalize()
    ws2 = rb.DweightWorkspace(150, H); ws2.begin()
    rb.rmsnorm_bwd_dweight_contrib(xp, dp, H, cl, 1e-6, ws2)
    dw2 = ws2.finalize()
    cl_np = rb.call_layout(np.arange(150, dtype=np.int32), 1, 150, with_plan=False)
    dx2 = rb.rmsnorm_bwd_dx(xp, w, dp, cl_np, 1e-6)
    assert torch.equal(dw1.view(torch.int32), dw2.view(torch.int32))
    assert torch.equal(dx1.view(torch.int16), dx2.view(torch.int16))
    # the forward without a plan equals the forward with one
    y1 = rb.rmsnorm_fwd(xp, w, cl, 1e-6)
    y2 = rb.rmsnorm_fwd(xp, w, cl_np, 1e-6)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert ws1.status() == 0 and ws2.status() == 0


def test_in_place_forward_and_dx_over_dy():
    H = 5120
    wl = _workload([33], H)
    x, dy, w = G.logical_inputs(wl)
    xp, dp = x.reshape(33, H).clone(), dy.reshape(33, H).clone()
    cl = rb.call_layout(np.arange(33, dtype=np.int32), 1, 33, with_plan=False)
    y_ref = rb.rmsnorm_fwd(xp, w, cl, 1e-6)
    dx_ref = rb.rmsnorm_bwd_dx(xp, w, dp, cl, 1e-6)
    d2 = dp.clone()
    rb.rmsnorm_bwd_dx(xp, w, d2, cl, 1e-6, dx=d2)
    x2 = xp.clone()
    rb.rmsnorm_fwd(x2, w, cl, 1e-6, y=x2)
    assert torch.equal(x2.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(d2.view(torch.int16), dx_ref.view(torch.int16))


def test_rstd_output_matches_oracle():
    H = 256
    wl = _workload([20, 12], H)
    x, dy, w = G.logical_inputs(wl)
    tok = np.array([3, -1, 0, 1, 2] + list(range(4, 32)), dtype=np.int32)
    cl = rb.call_layout(tok, 1, 32, with_plan=False)
    xp = torch.zeros(tok.size, H, dtype=torch.bfloat16, device=DEV)
    act = torch.as_tensor(tok >= 0, device=DEV)
    xp[act] = x.reshape(32, H)[torch.as_tensor(tok[tok >= 0], device=DEV).long()]
    rstd = torch.full((tok.size,), -7.0, device=DEV)
    rb.rmsnorm_fwd(xp, w, cl, 1e-6, rstd=rstd)
    _, ref = oracle.forward(x.reshape(32, H).cpu(), w.cpu(), 1e-6)
    got = rstd.cpu().numpy()
    assert got[1] == -7.0
    np.testing.assert_allclose(got[tok >= 0], ref[tok[tok >= 0]], rtol=2e-6)


# ------------------------------------------------------------------ status word

def test_double_and_missing_contributions_are_reported():
    H = 128
    wl = _workload([100], H)
    x, dy, w = G.logical_inputs(wl)
    xp, dp = x.reshape(100, H), dy.reshape(100, H)
    full = rb.call_layout(np.arange(100, dtype=np.int32), 1, 100)
    part = rb.call_layout(np.arange(10, dtype=np.int32), 1, 100)
    ws = rb.DweightWorkspace(100, H); ws.begin()
    rb.rmsnorm_bwd_dx(xp, w, dp, full, 1e-6, workspace=ws)
    rb.rmsnorm_bwd_dx(xp, w, dp, part, 1e-6, workspace=ws)       # rows 0..9 again
    ws.finalize()
    assert ws.status() & rb.STATUS_DOUBLE
    ws2 = rb.DweightWorkspace(100, H); ws2.begin()
    rb.rmsnorm_bwd_dx(xp, w, dp, part, 1e-6, workspace=ws2)      # rows 10..99 never arrive
    ws2.finalize()
    assert ws2.status() & rb.STATUS_MISSING
    ws3 = rb.DweightWorkspace(100, H); ws3.begin()
    rb.rmsnorm_bwd_dx(xp, w, dp, full, 1e-6, workspace=ws3)
    ws3.finalize()
    assert ws3.status() == 0


def test_workspace_for_other_sizes_is_reported():
    H = 128
    ws = rb.DweightWorkspace(100, H)
    ws.begin()
    lib = rb._load()
    import ctypes
    out = torch.empty(H, device=DEV)
    # finalize as if the workspace had been begun for 90 rows
    rc = lib.dweight_finalize(ctypes.c_void_p(ws.buf.data_ptr()), 90, H, ctypes.c_void_p(out.data_ptr()),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    assert ws.status() & rb.STATUS_HEADER

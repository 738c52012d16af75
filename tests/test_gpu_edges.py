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

@pytest.mark.parametrize("hidden", [8, 24, 128, 200, 4096, 5120])
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


def _exact_tree_inputs(n_tok, rpt, hidden, seed):
    """Inputs whose dweight leaves are exact and whose FP32 sums depend on the
    association order: eps = 0, every row of constant magnitude 2^k (so rstd =
    2^-k and xhat = +-1 exactly) and dy drawn from values that straddle 2^24.
    Returns bf16 x, dy [n_tok, rpt, hidden] and the tree replay of the leaves
    in logical row order (token-major, head-minor: row g*rpt + head)."""
    rng = np.random.default_rng(seed)
    n_rows = n_tok * rpt
    signs = rng.choice(np.array([-1.0, 1.0], dtype=np.float32), size=(n_rows, hidden))
    mags = (2.0 ** rng.integers(-3, 4, size=(n_rows, 1))).astype(np.float32)
    pool = np.array([16777216.0, 1.0, -1.0, 3.0, -16777216.0, 0.5, 2.0 ** -20, 65536.0, -0.0, 255.0],
                    dtype=np.float32)
    dy = pool[rng.integers(0, pool.size, size=(n_rows, hidden))]
    want = tree_replay.dweight(dy * signs)
    x = bf16(signs * mags).reshape(n_tok, rpt, hidden)
    return x, bf16(dy).reshape(n_tok, rpt, hidden), want


def _split_lengths(n, seed):
    """n tokens as a few samples of uneven length (at least one token each)."""
    rng = np.random.default_rng(seed)
    k = int(min(n, 1 + rng.integers(1, 7)))
    cuts = np.sort(rng.choice(np.arange(1, n), size=k - 1, replace=False)) if k > 1 else np.zeros(0, int)
    return np.diff(np.concatenate([[0], cuts, [n]])).astype(np.int64)


_TREE_KINDS = ("full", "chunked", "singleton", "padded_right", "padded_left", "permuted",
               "padded_right_chunked", "permuted_chunked")


def _assert_tree_layouts(lengths, rpt, hidden, seed, kinds=_TREE_KINDS, chunk=37):
    n_tok = int(np.sum(lengths))
    x, dy, want = _exact_tree_inputs(n_tok, rpt, hidden, seed)
    perm = synth.seeded_permutation(seed, len(lengths))
    ones = bf16(np.ones(hidden))
    for kind in kinds:
        lay = L.make_layout(kind, lengths, chunk=chunk, perm=perm)
        run = harness.run_layout(lay, x, dy, ones, 0.0, rows_per_token=rpt)
        assert run.status == 0, (kind, run.status)
        got = run.dweight.cpu().numpy()
        assert got.tobytes() == want.tobytes(), (kind, hidden, rpt, np.flatnonzero(got != want)[:5])


@pytest.mark.parametrize("hidden", [8192, 10240, 16384])
@pytest.mark.parametrize("n_tok", [1, 65, 259, 4999])
def test_dweight_tree_bitwise_on_cluster_kernels(hidden, n_tok):
    """Hidden sizes above 5120 run on 2- and 4-CTA clusters (row sums exchanged
    through distributed shared memory, column slices split over the CTAs;
    10240: 768-thread CTAs, whose column threads keep part of the unit tree
    in tensor memory); the tree must still be the fixed one, in every layout.
    4999 rows: 316 quarter units leave a partial last round, which the
    backward splits into eighths."""
    _assert_tree_layouts(_split_lengths(n_tok, hidden + n_tok), 1, hidden, hidden * 7 + n_tok)


@pytest.mark.parametrize("rpt", [8, 32])
@pytest.mark.parametrize("n_tok", [1, 7, 9, 100, 700])
def test_dweight_tree_bitwise_per_head_rows(rpt, n_tok):
    """Per-head norms (head_dim 128): logical row g*heads + head, so a token's
    heads are adjacent leaves and a 64-row block holds 64/heads tokens."""
    _assert_tree_layouts(_split_lengths(n_tok, rpt + n_tok), rpt, 128, rpt * 1000 + n_tok)


@pytest.mark.parametrize("hidden", [8, 128, 4096, 5120, 8192])
@pytest.mark.parametrize("chunk", [37, 16, 61])
def test_dweight_tree_bitwise_padded_and_permuted_layouts(hidden, chunk):
    """Several samples, padded on either side, permuted, and chunked so that
    call boundaries cut logical blocks at every offset (37 and 61 are prime to
    64; chunks of 16 cut the padded stream on quarter boundaries that are not
    logical ones)."""
    lengths = np.array([70, 3, 130, 1, 64, 9, 500, 37, 129])
    _assert_tree_layouts(lengths, 1, hidden, hidden + chunk, chunk=chunk)


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

@pytest.mark.parametrize("hidden", [8, 16, 24, 40, 64, 72, 128, 136, 200, 256, 264, 512, 1024, 4096, 4104, 5120,
                                    6144, 8192, 10240, 12288, 16384])
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

@pytest.mark.parametrize("H", [4096, 5120, 10240])
def test_contrib_only_and_dx_only_match_fused(H):
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


@pytest.mark.parametrize("with_plan", [False, True])
@pytest.mark.parametrize("H", [8, 64, 128, 256, 1024, 8192])
def test_rstd_output_matches_oracle(H, with_plan):
    """rstd of every active slot (small-row teams of 1 to 32 lanes, one CTA and
    2-CTA clusters); an inactive slot keeps what the caller put there."""
    wl = _workload([20, 12], H)
    x, dy, w = G.logical_inputs(wl)
    tok = np.array([3, -1, 0, 1, 2] + list(range(4, 32)), dtype=np.int32)
    cl = rb.call_layout(tok, 1, 32, with_plan=with_plan)
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

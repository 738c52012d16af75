"""GPU: sharded weight gradient over simulated ranks on one device.

Each simulated rank owns the logical tokens of its block ranges, runs its own
physical layout of them (different chunk sizes and a reversed call order per
rank) into its own workspace with local ids, and reduces its ranges to
nodes of the tree.  The all-gather goes through host memory; every rank then
combines the same roots.  The result must equal one device's dweight over
one packed call bit for bit, and match the FP64 oracle.
"""
import numpy as np
import pytest
import torch

import gpu_common as G
import synth
from invariant_rmsnorm_fwd_gb300 import sharded as S
import invariant_rmsnorm_fwd_gb300 as rb

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _calls(n_tok, chunk, rng):
    ids = np.arange(n_tok, dtype=np.int32)
    calls = [ids[i:i + chunk] for i in range(0, n_tok, chunk)]
    if len(calls) > 1 and rng.random() < 0.5:
        calls = calls[::-1]
    return calls


def _rank_backward(x, dy, w, eps, plan, rank, rng):
    """One rank: local workspace over its rows, its own layout, its roots."""
    R, H = plan.rows_per_token, w.shape[0]
    t0, t1 = plan.tokens(rank)
    n_loc = t1 - t0
    ws = rb.DweightWorkspace(n_loc * R, H)
    ws.begin()
    xl = x[t0:t1].reshape(n_loc, R, H)
    dl = dy[t0:t1].reshape(n_loc, R, H)
    chunk = int(rng.integers(1, max(2, n_loc)) if n_loc > 1 else 1)
    for tok in _calls(n_loc, chunk, rng):
        cl = rb.call_layout(tok, R, n_loc)
        idx = torch.as_tensor(tok, device="cuda").long()
        rb.rmsnorm_bwd_dx(xl[idx].contiguous(), w, dl[idx].contiguous(), cl, eps, workspace=ws)
    roots = S.local_roots(ws, plan, rank)
    assert ws.status() == 0
    return roots


def _single_device(x, dy, w, eps, R):
    H = w.shape[0]
    n_tok = x.shape[0]
    ws = rb.DweightWorkspace(n_tok * R, H)
    ws.begin()
    cl = rb.call_layout(np.arange(n_tok, dtype=np.int32), R, n_tok)
    rb.rmsnorm_bwd_dx(x.reshape(n_tok, R, H), w, dy.reshape(n_tok, R, H), cl, eps, workspace=ws)
    return ws, ws.finalize()


@pytest.mark.parametrize("cfg,world,rpr", [("c0", 2, 4), ("c0", 8, 1), ("c1", 1, 4), ("c1", 2, 4), ("c1", 3, 2),
                                           ("c1", 8, 4), ("c1", 5, 1)])
def test_simulated_ranks_equal_one_device(cfg, world, rpr):
    wl = synth.config(cfg)
    x, dy, w = G.logical_inputs(wl)
    plan = S.plan_shards(wl.n_tokens, 1, world, ranges_per_rank=rpr)
    rng = np.random.default_rng(world * 100 + rpr)
    per = [_rank_backward(x, dy, w, wl.eps, plan, r, rng) for r in range(world)]
    host = [p.cpu() for p in per]                           # the all-gather, through host memory
    roots = S.assemble_roots(host, plan).cuda()
    dw = rb.dweight_combine(roots)
    _, want = _single_device(x, dy, w, wl.eps, 1)
    assert torch.equal(dw.view(torch.int32), want.view(torch.int32))


def test_qk_heads_sharded_over_four_ranks():
    wl = synth.config("c3")
    R = wl.heads[1]                                          # K: 8 rows per token
    x, dy, w = G.logical_inputs(wl, head_set=1, rpt=R)
    plan = S.plan_shards(wl.n_tokens, R, 4)
    rng = np.random.default_rng(5)
    per = [_rank_backward(x, dy, w, wl.eps, plan, r, rng).cpu() for r in range(4)]
    dw = rb.dweight_combine(S.assemble_roots(per, plan).cuda())
    _, want = _single_device(x, dy, w, wl.eps, R)
    assert torch.equal(dw.view(torch.int32), want.view(torch.int32))


@pytest.mark.parametrize("n_rows", [1, 64, 65, 200, 4096 + 64 * 3 + 5])
def test_ranges_of_a_global_workspace_are_nodes(n_rows):
    """finalize_range over a global workspace, then combine, equals finalize."""
    H = 256
    wl = synth.Workload("t", H, np.asarray([n_rows]), seed=n_rows, chunk_rows=37)
    x, dy, w = G.logical_inputs(wl)
    ws, want = _single_device(x, dy, w, wl.eps, 1)
    nb = (n_rows + 63) // 64
    for bc in (1, 2, 4, 16, 64):
        roots = torch.stack([ws.finalize_range(lo, bc) for lo in range(0, nb, bc)])
        got = rb.dweight_combine(roots)
        assert torch.equal(got.view(torch.int32), want.view(torch.int32)), bc
    assert ws.status() == 0


def test_bad_ranges_and_roots_are_refused():
    H = 128
    ws = rb.DweightWorkspace(64 * 6, H)
    ws.begin()
    for lo, cnt in ((1, 2), (0, 3), (6, 1), (-2, 2), (0, 0)):
        with pytest.raises(rb.RmsNormError):
            ws.finalize_range(lo, cnt)
    with pytest.raises(rb.RmsNormError):
        rb.dweight_combine(torch.zeros(0, H, device="cuda"))
    with pytest.raises(rb.RmsNormError):
        rb.dweight_combine(torch.zeros(2048, H, device="cuda"))


def test_sharded_result_matches_oracle():
    wl = synth.config("c1")
    x, dy, w = G.logical_inputs(wl)
    plan = S.plan_shards(wl.n_tokens, 1, 4)
    rng = np.random.default_rng(1)
    per = [_rank_backward(x, dy, w, wl.eps, plan, r, rng).cpu() for r in range(4)]
    dw = rb.dweight_combine(S.assemble_roots(per, plan).cuda())
    import oracle
    import tolerances as tol
    H = wl.hidden
    _, _, dw_ref, s_scale = oracle.backward(x.reshape(-1, H).cpu(), w.cpu(), dy.reshape(-1, H).cpu(), wl.eps,
                                            want_dx=False)
    r = tol.check("dweight", dw.cpu().numpy(), dw_ref, tol.bound_dw(dw_ref, s_scale))
    assert r["violations"] == 0, r

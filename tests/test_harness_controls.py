"""Falsifiability of the invariance harness (CPU, synthetic operators).

"WS1 C4 (#270) closeout evidence", section "The matrix is falsifiable": a
layout-sensitive operator must be judged red, an operator that depends only
on logical identity must be judged green, and the layouts must really
differ.  The layout-sensitive operator here is the failure the same page
documents ("Historical finding - RMSNorm dweight is not chunk/batch
decomposable"): a left fold of the rows of each call, the call results added
in call order.  A left fold over 59 rows is not bitwise equal to the sum of
left folds over 11 + 16 + 13 + 19 rows.
"""
import numpy as np
import torch

import synth
from invariant_rmsnorm_fwd_gb300 import harness
from invariant_rmsnorm_fwd_gb300 import layout as L
from oracle import tree_replay


def _leaves(n, H, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(n, H)) * np.exp(rng.normal(size=(n, 1)) * 3)).astype(np.float32)


def _left_fold_per_call(lay, leaves):
    total = np.zeros(leaves.shape[1], np.float32)
    for tok in lay.calls:
        acc = np.zeros(leaves.shape[1], np.float32)
        for t in tok:                                      # physical order, padding skipped
            if t >= 0:
                acc = (acc + leaves[t]).astype(np.float32)
        total = (total + acc).astype(np.float32)
    return total


def _run(name, dweight, y=None):
    H = dweight.shape[0]
    y = torch.zeros(1, H, dtype=torch.bfloat16) if y is None else y
    return harness.LayoutRun(name, y, y.clone(), torch.as_tensor(dweight), 0, 1, [1])


def test_pages_failure_mechanism_is_judged_red():
    wl = synth.config("c0p")
    lays = L.workload_layouts(wl)
    leaves = _leaves(59, 8)
    runs = {k: _run(k, _left_fold_per_call(v, leaves)) for k, v in lays.items()}
    rep = harness.assert_batch_invariant(runs, lays)
    assert not rep.green
    f = rep.first_failure()
    assert f.tensor == "dweight" and f.max_abs > 0
    # the singleton aggregate (11 + 16 + 13 + 19) differs from one left fold over 59
    assert not np.array_equal(_left_fold_per_call(lays["singleton"], leaves),
                              _left_fold_per_call(lays["full"], leaves))


def test_logical_order_tree_is_judged_green():
    wl = synth.config("c0p")
    lays = L.workload_layouts(wl)
    leaves = _leaves(59, 8)
    runs = {k: _run(k, tree_replay.dweight(leaves)) for k in lays}
    rep = harness.assert_batch_invariant(runs, lays)
    assert rep.green, rep.summary()


def test_identical_layouts_are_not_accepted_as_evidence():
    wl = synth.config("c0p")
    lays = L.workload_layouts(wl)
    same = {k: lays["full"] for k in lays}
    same = {k: L.Layout(k, v.calls, v.n_logical_tokens) for k, v in same.items()}
    leaves = _leaves(59, 8)
    runs = {k: _run(k, tree_replay.dweight(leaves)) for k in same}
    rep = harness.assert_batch_invariant(runs, same)
    assert not rep.green and not any(rep.distinct.values())


def test_padding_leak_is_judged_red():
    wl = synth.config("c0p")
    lays = L.workload_layouts(wl)
    leaves = _leaves(59, 8)
    runs = {k: _run(k, tree_replay.dweight(leaves)) for k in lays}
    bad = tree_replay.dweight(leaves).copy()
    bad[3] = np.nan                                        # a NaN padding row reached the sum
    runs["padded_left"] = _run("padded_left", bad)
    rep = harness.assert_batch_invariant(runs, lays)
    assert not rep.green and rep.first_failure().layout == "padded_left"


def test_nonzero_status_is_red():
    wl = synth.config("c0p")
    lays = L.workload_layouts(wl)
    leaves = _leaves(59, 8)
    runs = {k: _run(k, tree_replay.dweight(leaves)) for k in lays}
    runs["chunked"].status = 2
    assert not harness.assert_batch_invariant(runs, lays).green


def test_drift_attribution_metrics():
    a = torch.tensor([[1.0, 2.0, 3.0, 4.0], [5.0, 6.0, 7.0, 8.0]])
    b = a.clone()
    b[1, 2] = 7.5                                          # one element of logical row 1 drifts by 0.5
    d = harness.bitwise_diff("dweight", a, b, "chunked", "full")
    assert not d.equal and d.mismatches == 1 and d.first_logical_index == 1
    assert d.max_abs == 0.5 and abs(d.mean_abs - 0.5 / 8) < 1e-12
    assert 0.0 <= d.p99_abs <= 0.5
    same = harness.bitwise_diff("dweight", a, a.clone(), "chunked", "full")
    assert same.equal and same.mismatches == 0 and same.max_abs == 0.0
    # bit patterns decide: -0.0 differs from +0.0
    z = harness.bitwise_diff("dweight", torch.tensor([-0.0]), torch.tensor([0.0]), "x", "y")
    assert not z.equal and z.max_abs == 0.0

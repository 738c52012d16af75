"""GPU: accuracy against the FP64 oracle and bitwise invariance across layouts.

Every workload runs in the six layout cells (full, chunked, singleton,
right/left padded, permuted) plus its headline layout, through the C ABI.
Outputs restored to logical order must be bit-identical across layouts and
within the stated tolerances of the oracle; padding rows must stay untouched
and the device status word must be clear.
"""
import numpy as np
import pytest
import torch

import gpu_common as G
import synth
from invariant_rmsnorm_fwd_gb300 import harness

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _assert_green(rep, runs):
    s = rep.summary()
    assert rep.green, s
    for name, r in runs.items():
        assert r.untouched_padding, name


def _assert_accurate(reports):
    for r in reports:
        assert r["violations"] == 0, r


@pytest.mark.parametrize("cfg", ["c0", "c0p", "c1"])
def test_invariance_and_accuracy(cfg):
    wl = synth.config(cfg)
    x, dy, w, lays, runs = G.run_all_layouts(wl)
    rep = harness.assert_batch_invariant(runs, lays)
    _assert_green(rep, runs)
    for name in ("full", "chunked"):
        _assert_accurate(G.oracle_check(runs[name], x, dy, w, wl.eps))


def test_c2_hidden8192_padded_chunked():
    wl = synth.config("c2")
    x, dy, w, lays, runs = G.run_all_layouts(wl, kinds=["full", "padded_right_chunked", "singleton",
                                                          "padded_right", "padded_left", "permuted", "chunked"])
    _assert_green(harness.assert_batch_invariant(runs, lays), runs)
    _assert_accurate(G.oracle_check(runs["padded_right_chunked"], x, dy, w, wl.eps))


@pytest.mark.parametrize("head_set,heads", [(0, 32), (1, 8)])
def test_c3_per_head_norm(head_set, heads):
    wl = synth.config("c3")
    x, dy, w, lays, runs = G.run_all_layouts(wl, head_set=head_set, rpt=heads)
    _assert_green(harness.assert_batch_invariant(runs, lays), runs)
    _assert_accurate(G.oracle_check(runs["chunked"], x, dy, w, wl.eps))


def test_c4_hidden5120_slots_quarter_density():
    wl = synth.config("c4")
    x, dy, w, lays, runs = G.run_all_layouts(wl, kinds=["full", "permuted_slots_left_chunked", "singleton",
                                                          "padded_right", "padded_left", "permuted", "chunked"])
    _assert_green(harness.assert_batch_invariant(runs, lays), runs)
    _assert_accurate(G.oracle_check(runs["permuted_slots_left_chunked"], x, dy, w, wl.eps))


def test_repeatable_run_to_run():
    wl = synth.config("c1")
    x, dy, w, lays, runs = G.run_all_layouts(wl, kinds=["full", "chunked"])
    again = harness.run_layout(lays["chunked"], x, dy, w, wl.eps)
    for t in ("y", "dx", "dweight"):
        assert harness.bitwise_diff(t, getattr(again, t), getattr(runs["chunked"], t), "again", "chunked").equal

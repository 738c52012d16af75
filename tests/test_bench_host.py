"""Host-side pieces of the bench (CPU): the recorded-traffic gate and cut workloads."""
import importlib.util
import json
import os

import numpy as np

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_recorded_traffic_is_used_only_for_its_workload_and_sources():
    b = _bench()
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for rec in d.get("records", [d]):
        got = b.recorded_traffic(rec["workload"], rec["layout"])
        if rec["source_sha256"] == b.source_sha256():
            assert got == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        else:
            assert got is None                            # sources changed since the capture
        assert b.recorded_traffic(rec["workload"], "no-such-layout") is None
    assert b.recorded_traffic("c9", "full") is None


def test_truncated_workload_keeps_the_first_tokens_and_values():
    wl = synth.config("c1")
    cut = synth.truncated(wl, 5000)
    assert cut.n_tokens == 5000 and cut.hidden == wl.hidden
    assert np.array_equal(cut.lengths[:-1], wl.lengths[:len(cut.lengths) - 1])
    assert cut.lengths[-1] <= wl.lengths[len(cut.lengths) - 1]
    # values are keyed by logical id: the first rows are the same
    a = synth.logical_tensor(wl, synth.TAG_X, 16, wl.x_std)
    c = synth.logical_tensor(cut, synth.TAG_X, 16, cut.x_std)
    assert np.array_equal(a.float().numpy(), c.float().numpy())


def test_parse_defaults_run_one_gpu_briefly():
    import sys
    b = _bench()
    old = sys.argv
    try:
        sys.argv = ["bench.py"]
        args = b.parse()
    finally:
        sys.argv = old
    assert args.gpus == 1 and args.steps >= 1 and args.warmup >= 3 and args.impl == "ours"
    assert args.config == "c4" and not args.chain and not args.gemm
    assert set(args.also.split(",")) == {"c1", "c2", "c3"}


def test_e2e_subcalls_cover_every_token_once_and_ramp():
    from invariant_rmsnorm_fwd_gb300 import layout as L
    b = _bench()
    for cfg, kind in (("c1", "full"), ("c2", "padded_right_chunked"), ("c4", "permuted_slots_left_chunked"),
                      ("c0", "padded_left")):
        wl = synth.config(cfg)
        lay = L.workload_layouts(wl, kinds=[kind])[kind]
        subs = b.e2e_subcalls(lay, 4096, 1024)
        ids = np.concatenate([t[t >= 0] for t in subs])
        assert np.array_equal(np.sort(ids), np.arange(wl.n_tokens))
        assert all(t.size <= 4096 and t[0] >= 0 and t[-1] >= 0 for t in subs)
        # padding dropped at the ends only: the slots kept are contiguous pieces of the calls
        n_pad = sum(int((t < 0).sum()) for t in subs)
        assert n_pad <= sum(int((c < 0).sum()) for c in lay.calls)
    wl = synth.config("c1")
    sizes = [t.size for t in b.e2e_subcalls(L.workload_layouts(wl, kinds=["full"])["full"], 4096, 1024)]
    assert sizes[:3] == [1024, 2048, 4096] and sum(sizes) == wl.n_tokens

"""Layout mapper and host planner (CPU only)."""
import json
import os

import numpy as np
import pytest

import synth
from invariant_rmsnorm_fwd_gb300 import layout as L
from invariant_rmsnorm_fwd_gb300.harness import layouts_differ

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_pages_worked_layout_table_is_reproduced():
    g = json.load(open(os.path.join(GOLD, "pages_layout.json")))
    wl = synth.config("c0p")
    assert list(wl.lengths) == g["sample_lengths"] and wl.hidden == g["hidden"]
    lays = L.workload_layouts(wl)
    for cell, want in g["cells"].items():
        if cell == "singleton_s0":
            lay = lays["singleton"]
            assert lay.rows_per_call[0] == want["rows"][0]
            assert len(lay.calls) == len(wl.lengths)
            continue
        lay = lays[cell]
        assert len(lay.calls) == want["calls"], cell
        assert lay.rows_per_call == want["rows"], cell


def test_c0_chunk_boundaries_over_packed_stream():
    lay = L.workload_layouts(synth.config("c0"))["chunked"]
    assert list(np.cumsum(lay.rows_per_call)) == [7, 11, 18, 25, 27, 34, 40, 47, 54, 59]
    assert L.workload_layouts(synth.config("c0"))["padded_right"].rows_per_call == [80]


@pytest.mark.parametrize("cfg", ["c0", "c0p", "c1", "c2", "c3", "c4"])
def test_every_layout_is_a_partition_and_differs_from_full(cfg):
    wl = synth.config(cfg)
    lays = L.workload_layouts(wl)
    for name, lay in lays.items():
        lay.check_partition()
        if name != "full":
            assert layouts_differ(lays["full"], lay), name


def test_logical_id_is_layout_independent():
    lengths = np.array([3, 1, 2])
    perm = L.make_layout("permuted", lengths, perm=np.array([2, 0, 1]))
    assert list(perm.calls[0]) == [4, 5, 0, 1, 2, 3]
    left = L.make_layout("padded_left", lengths, slot=3)
    assert list(left.calls[0]) == [0, 1, 2, -1, -1, 3, -1, 4, 5]


def test_partition_check_rejects_duplicates():
    lay = L.Layout("bad", [np.array([0, 1], np.int32), np.array([1, 2], np.int32)], 3)
    with pytest.raises(ValueError):
        lay.check_partition()


# ------------------------------------------------------------------ planner

def _items(buf, n):
    a = np.frombuffer(buf.tobytes(), dtype=np.int32).reshape(n, 132)
    return a[:, 0], a[:, 1], a[:, 2], a[:, 4:68], a[:, 68:132]


def _plan(tok, rpt, ntok):
    import invariant_rmsnorm_fwd_gb300 as rb
    return rb.plan_build(tok, rpt, ntok)


@pytest.mark.parametrize("cfg,kind,rpt", [("c0", "chunked", 1), ("c0", "padded_left", 1), ("c0p", "singleton", 1),
                                          ("c1", "chunked", 1), ("c2", "padded_right_chunked", 1),
                                          ("c3", "chunked", 32), ("c4", "permuted_slots_left_chunked", 1)])
def test_plan_covers_every_active_row_once(cfg, kind, rpt):
    wl = synth.config(cfg)
    lay = L.workload_layouts(wl, kinds=[kind])[kind]
    N = wl.n_tokens * rpt
    seen = np.zeros(N, dtype=np.int64)
    whole_blocks = []
    for tok in lay.calls[:40]:
        buf, n, whole, spill = _plan(tok, rpt, wl.n_tokens)
        kind_a, block, count, prow, lrow = _items(buf, n)
        n_sp_items = (spill + 63) // 64
        assert np.all(kind_a[:whole] == 0) and np.all(kind_a[n - n_sp_items:] == 1)
        assert np.all(kind_a[whole:n - n_sp_items] == 2)
        for i in range(n):
            used = lrow[i][lrow[i] >= 0]
            pr = prow[i][lrow[i] >= 0]
            assert used.size == count[i]
            # physical row -> token slot -> logical id agrees with the plan
            assert np.array_equal(tok[pr // rpt].astype(np.int64) * rpt + pr % rpt, used)
            seen[used] += 1
            if kind_a[i] == 0:
                b = block[i]
                assert np.array_equal(used, np.arange(b * 64, min(b * 64 + 64, N)))
                whole_blocks.append(b)
            if kind_a[i] == 2:                        # complete quarters of a cut block, each row at its place
                b = block[i]
                slots = np.nonzero(lrow[i] >= 0)[0]
                assert np.array_equal(lrow[i][slots], b * 64 + slots)
                mask = np.frombuffer(buf.tobytes(), dtype=np.int32).reshape(n, 132)[i, 3]
                for q in range(4):
                    q_rows = np.arange(b * 64 + 16 * q, min(b * 64 + 16 * q + 16, N))
                    if (mask >> q) & 1:
                        assert q_rows.size and np.isin(q_rows, used).all()
                    else:
                        assert not np.isin(q_rows, used).any()
        assert int(np.sum(count[n - n_sp_items:])) == spill
    assert seen.max() <= 1
    assert len(set(whole_blocks)) == len(whole_blocks)


def test_plan_whole_vs_cut_blocks():
    tok = np.arange(0, 130, dtype=np.int32)              # ids 0..129 of N=200: blocks 0,1 whole, block 2 cut
    buf, n, whole, spill = _plan(tok, 1, 200)
    assert (n, whole, spill) == (3, 2, 2)
    tok = np.arange(0, 150, dtype=np.int32)              # block 2 cut after its first quarter (128..143) and 6 rows
    buf, n, whole, spill = _plan(tok, 1, 200)
    assert (n, whole, spill) == (4, 2, 6)
    kind_a, block, count, prow, lrow = _items(buf, n)
    assert list(kind_a) == [0, 0, 2, 1] and block[2] == 2 and count[2] == 16
    assert np.frombuffer(buf.tobytes(), dtype=np.int32).reshape(n, 132)[2, 3] == 0b0001
    tok = np.arange(190, 200, dtype=np.int32)            # block 2's last 2 rows, block 3 (192..199) whole
    buf, n, whole, spill = _plan(tok, 1, 200)
    assert (n, whole, spill) == (2, 1, 2)
    tok = np.arange(176, 199, dtype=np.int32)            # block 2's last quarter; block 3 cut short of row 199
    buf, n, whole, spill = _plan(tok, 1, 200)
    assert (n, whole, spill) == (2, 0, 7)
    tok = np.arange(128, 200, dtype=np.int32)            # block 2 (128..191) whole, block 3 (192..199) whole
    buf, n, whole, spill = _plan(tok, 1, 200)
    assert (whole, spill) == (2, 0)


def test_plan_rejects_bad_ids():
    import invariant_rmsnorm_fwd_gb300 as rb
    with pytest.raises(rb.RmsNormError) as e:
        _plan(np.array([0, 1, 1], np.int32), 1, 5)
    assert e.value.code == -9
    with pytest.raises(rb.RmsNormError) as e:
        _plan(np.array([0, 5], np.int32), 1, 5)
    assert e.value.code == -8
    with pytest.raises(rb.RmsNormError):
        _plan(np.array([-2], np.int32), 1, 5)


def test_plan_is_a_function_of_the_ids_only():
    tok = synth.seeded_permutation(3, 300).astype(np.int32)
    a = _plan(tok, 1, 300)[0]
    b = _plan(tok.copy(), 1, 300)[0]
    assert np.array_equal(a, b)


def _plan_ref(tok, rpt, ntok):
    """The plan spelled out in numpy: active rows in logical order, one item per
    logical block held whole (its rows in order, -1 beyond the block's last row),
    the rows of cut blocks in logical order cut into items of 64."""
    act = np.nonzero(tok >= 0)[0]
    order = act[np.argsort(tok[act], kind="stable")]
    lrows = (tok[order].astype(np.int64)[:, None] * rpt + np.arange(rpt)).ravel()
    prows = (order.astype(np.int64)[:, None] * rpt + np.arange(rpt)).ravel()
    n_rows = ntok * rpt
    whole, quarter, sp_l, sp_p = [], [], [], []
    for b in np.unique(lrows // 64):
        sel = lrows // 64 == b
        if sel.sum() == min(64, n_rows - 64 * b):
            whole.append((0, b, prows[sel], lrows[sel]))
            continue
        mask, slots, qp = 0, [], []
        for q in range(4):
            q_rows = np.arange(64 * b + 16 * q, min(64 * b + 16 * q + 16, n_rows))
            inq = sel & (lrows // 16 == 4 * b + q)
            if q_rows.size and inq.sum() == q_rows.size:
                mask |= 1 << q
                slots.append(lrows[inq] - 64 * b)
                qp.append((prows[inq], lrows[inq]))
            elif inq.any():
                sp_l.append(lrows[inq])
                sp_p.append(prows[inq])
        if mask:
            quarter.append((b, mask, qp))
    sp_l = np.concatenate(sp_l) if sp_l else np.zeros(0, np.int64)
    sp_p = np.concatenate(sp_p) if sp_p else np.zeros(0, np.int64)
    items = [(k, b, p, l, 0) for k, b, p, l in whole]
    for b, mask, qp in quarter:
        p64 = np.full(64, -1, np.int64)
        l64 = np.full(64, -1, np.int64)
        for p, l in qp:
            p64[l - 64 * b] = p
            l64[l - 64 * b] = l
        items.append((2, b, p64, l64, mask))
    items += [(1, -1, sp_p[k:k + 64], sp_l[k:k + 64], 0) for k in range(0, sp_l.size, 64)]
    out = np.full((len(items), 132), -1, dtype=np.int32)
    for i, (kind, b, p, l, mask) in enumerate(items):
        out[i, :4] = (kind, b, int((l >= 0).sum()), mask)
        out[i, 4:4 + p.size] = p
        out[i, 68:68 + l.size] = l
    return out, len(whole), int(sp_l.size)


@pytest.mark.parametrize("cfg,kind,rpt", [("c0", "permuted", 1), ("c0p", "padded_right", 3), ("c1", "chunked", 1),
                                          ("c1", "permuted", 1), ("c3", "singleton", 8),
                                          ("c4", "permuted_slots_left_chunked", 1)])
def test_plan_bytes_match_the_spelled_out_plan(cfg, kind, rpt):
    wl = synth.config(cfg)
    lay = L.workload_layouts(wl, kinds=[kind])[kind]
    calls = lay.calls[:12] + [np.ascontiguousarray(lay.calls[0][::-1])]      # a descending call too
    for tok in calls:
        buf, n, whole, spill = _plan(tok, rpt, wl.n_tokens)
        ref, ref_whole, ref_spill = _plan_ref(tok, rpt, wl.n_tokens)
        assert (n, whole, spill) == (ref.shape[0], ref_whole, ref_spill)
        assert np.array_equal(np.frombuffer(buf.tobytes(), dtype=np.int32).reshape(n, 132), ref)


def test_plan_into_caller_buffer_and_capacity():
    import invariant_rmsnorm_fwd_gb300 as rb
    tok = np.arange(0, 200, dtype=np.int32)               # N=200: three whole blocks and the short last one
    out = np.zeros(4 * rb.PLAN_ITEM_BYTES, dtype=np.uint8)
    buf, n, whole, spill = rb.plan_build(tok, 1, 200, out=out)
    assert (n, whole, spill) == (4, 4, 0) and np.shares_memory(buf, out)
    ref = _plan_ref(tok, 1, 200)[0]
    assert np.array_equal(np.frombuffer(out.tobytes(), dtype=np.int32).reshape(4, 132), ref)
    with pytest.raises(rb.RmsNormError) as e:
        rb.plan_build(tok, 1, 200, out=np.zeros(3 * rb.PLAN_ITEM_BYTES, dtype=np.uint8))
    assert e.value.code == -10
    with pytest.raises(ValueError):
        rb.plan_build(tok, 1, 200, out=np.zeros(4 * rb.PLAN_ITEM_BYTES, dtype=np.int32))


def test_plan_build_from_several_threads():
    """The planner keeps per-thread working arrays: concurrent calls (ctypes
    releases the GIL) must each get their own call's plan."""
    import concurrent.futures as cf
    wl = synth.config("c4")
    lay = L.workload_layouts(wl, kinds=["permuted_slots_left_chunked"])["permuted_slots_left_chunked"]
    calls = [c for c in lay.calls if (c >= 0).any()][:24]
    want = [_plan_ref(c, 1, wl.n_tokens)[0] for c in calls]

    def one(i):
        buf, n, _, _ = _plan(calls[i], 1, wl.n_tokens)
        return np.frombuffer(buf.tobytes(), dtype=np.int32).reshape(n, 132)

    with cf.ThreadPoolExecutor(8) as ex:
        for _ in range(3):
            got = list(ex.map(one, range(len(calls))))
            assert all(np.array_equal(g, w) for g, w in zip(got, want))

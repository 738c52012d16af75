"""GPU: deterministic weight gradient of a linear layer (det_gemm dW).

dW = sum_g dy_g^T x_g over the logical tokens must be bitwise identical for
every layout of the multiset, match the FP64 oracle within 1e-4 of the terms'
scale, be exact where every sum is exact, and report missing and doubled
tokens.  A per-call accumulation (the failure the pages document for det_gemm)
is shown to differ.
"""
import numpy as np
import pytest
import torch

import synth
import tolerances as tol
from oracle import gemm as ogemm
from invariant_rmsnorm_fwd_gb300 import harness
from invariant_rmsnorm_fwd_gb300 import layout as L
import invariant_rmsnorm_fwd_gb300 as rb

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _inputs(wl, I, O):
    wi = synth.Workload("x", I, wl.lengths, seed=wl.seed, x_std=wl.x_std, dy_std=wl.dy_std)
    wo = synth.Workload("dy", O, wl.lengths, seed=wl.seed, x_std=wl.x_std, dy_std=wl.dy_std)
    x = synth.logical_tensor(wi, synth.TAG_X, wl.n_tokens, wl.x_std, device="cuda")
    dy = synth.logical_tensor(wo, synth.TAG_DY, wl.n_tokens, wl.dy_std, device="cuda")
    return x, dy


@pytest.mark.parametrize("cfg,I,O", [("c0", 64, 128), ("c0p", 8, 8), ("c1", 512, 1024), ("c2", 256, 128)])
def test_layout_invariant_and_accurate(cfg, I, O):
    wl = synth.config(cfg)
    if wl.n_tokens > 20000:
        wl = synth.truncated(wl, 20000)
    x, dy = _inputs(wl, I, O)
    lays = L.workload_layouts(wl)
    runs = {k: harness.run_layout_gemm(v, x, dy) for k, v in lays.items()}
    rep = harness.assert_batch_invariant(runs, lays)
    assert rep.green, rep.summary()
    ref, s = ogemm.dw(x.cpu(), dy.cpu())
    r = tol.check("dW", runs["full"].dweight.cpu().numpy(), ref, tol.bound_dw(ref, s))
    assert r["violations"] == 0, r


@pytest.mark.parametrize("n,I,O", [(1000, 328, 200), (2000, 4096, 4096), (77, 8, 4104), (64, 264, 136)])
def test_tile_edges_and_many_tiles_per_cta(n, I, O):
    """dW tiles are 128 (o) x up to 256 (i) over slabs of 64 tokens: partial
    tiles in both directions, a token count that is not a multiple of 64, and
    (4096 x 4096) more tiles than CTAs, so each CTA alternates its two
    tensor-memory accumulators.  Chunked and permuted layouts must give the
    packed call's bits, and the oracle's values within tolerance."""
    lengths = np.array([n // 3, n - n // 3 - n // 5, n // 5]) if n >= 15 else np.array([n])
    lengths = lengths[lengths > 0]
    wl = synth.Workload("tiles", 8, lengths, seed=n + I + O, x_std=1.0, dy_std=1e-2, chunk_rows=37)
    x, dy = _inputs(wl, I, O)
    lays = L.workload_layouts(wl, kinds=["full", "chunked", "permuted"])
    runs = {k: harness.run_layout_gemm(v, x, dy) for k, v in lays.items()}
    rep = harness.assert_batch_invariant(runs, lays)
    assert rep.green, rep.summary()
    ref, s = ogemm.dw(x.cpu(), dy.cpu())
    r = tol.check("dW", runs["full"].dweight.cpu().numpy(), ref, tol.bound_dw(ref, s))
    assert r["violations"] == 0, r


def test_exact_sums_are_exact():
    """Small integers: every product and partial sum is exact in FP32, so the GPU
    result must equal the FP64 oracle bit for bit whatever its order."""
    rng = np.random.default_rng(9)
    n, I, O = 300, 64, 32
    x = torch.as_tensor(rng.integers(-4, 5, size=(n, I)).astype(np.float32)).to(torch.bfloat16).cuda()
    dy = torch.as_tensor(rng.integers(-4, 5, size=(n, O)).astype(np.float32)).to(torch.bfloat16).cuda()
    lay = L.make_layout("chunked", [n], chunk=37)
    run = harness.run_layout_gemm(lay, x, dy)
    ref, _ = ogemm.dw(x.cpu(), dy.cpu())
    assert np.array_equal(run.dweight.cpu().numpy().astype(np.float64), ref)
    assert run.status == 0


def test_scale_and_empty_multiset():
    n, I, O = 100, 16, 24
    x = torch.randn(n, I, device="cuda").to(torch.bfloat16)
    dy = torch.randn(n, O, device="cuda").to(torch.bfloat16)
    ws = rb.GemmDwWorkspace(n, I, O)
    ws.begin()
    ws.contrib(x, dy, rb.call_layout(np.arange(n, dtype=np.int32), 1, n, with_plan=False))
    d1 = ws.finalize()
    d2 = ws.finalize(grad_scale=0.5)                    # a power of two: exact scaling
    assert torch.equal((d1 * 0.5).view(torch.int32), d2.view(torch.int32))
    e = rb.GemmDwWorkspace(0, I, O)
    e.begin()
    assert torch.equal(e.finalize().cpu(), torch.zeros(O, I)) and e.status() == 0


def test_missing_double_and_bad_arguments():
    n, I, O = 50, 16, 16
    x = torch.randn(n, I, device="cuda").to(torch.bfloat16)
    dy = torch.randn(n, O, device="cuda").to(torch.bfloat16)
    ws = rb.GemmDwWorkspace(n, I, O)
    ws.begin()
    ws.contrib(x[:10], dy[:10], rb.call_layout(np.arange(10, dtype=np.int32), 1, n, with_plan=False))
    ws.finalize()
    assert ws.status() & rb.STATUS_MISSING
    ws.begin()
    full = rb.call_layout(np.arange(n, dtype=np.int32), 1, n, with_plan=False)
    ws.contrib(x, dy, full)
    ws.contrib(x, dy, full)
    ws.finalize()
    assert ws.status() & rb.STATUS_DOUBLE
    with pytest.raises(rb.RmsNormError) as e:
        ws.finalize(grad_scale=float("nan"))
    assert e.value.code == -13
    with pytest.raises(rb.RmsNormError) as e:                  # rows_per_token must be 1
        ws.contrib(x, dy, rb.CallLayout(full.tok_id, None, 0, n, 2, n))
    assert e.value.code == -5


def test_per_call_accumulation_is_not_invariant():
    """The failure class: summing per-call FP32 products in call order differs
    from the logical-order GEMM for random data."""
    wl = synth.config("c0p")
    x, dy = _inputs(wl, 64, 64)
    lays = L.workload_layouts(wl)
    per_call = torch.zeros(64, 64, device="cuda")
    for tok in lays["singleton"].calls:
        idx = torch.as_tensor(tok[tok >= 0], device="cuda").long()
        per_call = per_call + dy[idx].float().T @ x[idx].float()
    good = harness.run_layout_gemm(lays["full"], x, dy).dweight
    assert not torch.equal(per_call.view(torch.int32), good.view(torch.int32))

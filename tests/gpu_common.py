"""Helpers of the GPU tests: inputs from synth, outputs checked against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import tolerances as tol
from invariant_rmsnorm_fwd_gb300 import harness
from invariant_rmsnorm_fwd_gb300 import layout as L


def logical_inputs(wl, head_set: int = 0, rpt: int = 1, device="cuda"):
    n_rows = wl.n_tokens * rpt
    x = synth.logical_tensor(wl, synth.TAG_X, n_rows, wl.x_std, head_set, device=device)
    dy = synth.logical_tensor(wl, synth.TAG_DY, n_rows, wl.dy_std, head_set, device=device)
    w = synth.weight(wl, head_set, device=device)
    return x.reshape(wl.n_tokens, rpt, wl.hidden), dy.reshape(wl.n_tokens, rpt, wl.hidden), w


def sample_rows(n: int, k: int = 2048, seed: int = 0) -> np.ndarray:
    """All rows if n <= k, else first/last 64 rows plus a seeded sample."""
    if n <= k:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    pick = np.concatenate([np.arange(64), np.arange(n - 64, n), rng.choice(n, k - 128, replace=False)])
    return np.unique(pick)


def oracle_check(run: harness.LayoutRun, x, dy, w, eps: float, rows=None) -> list:
    """Compare a layout run (logical order) with the FP64 oracle; returns tolerance reports."""
    H = w.shape[0]
    xr = x.reshape(-1, H)
    dyr = dy.reshape(-1, H)
    n = xr.shape[0]
    rows = sample_rows(n) if rows is None else rows
    ridx = torch.as_tensor(rows, device=xr.device)
    xs, dys = xr[ridx].cpu(), dyr[ridx].cpu()
    wc = w.cpu()
    y_ref, _ = oracle.forward(xs, wc, eps)
    dx_ref, k_scale, _, _ = oracle.backward(xs, wc, dys, eps)
    _, _, dw_ref, s_scale = oracle.backward(xr.cpu(), wc, dyr.cpu(), eps, want_dx=False)
    y = run.y.reshape(-1, H)[ridx].float().cpu().numpy()
    dx = run.dx.reshape(-1, H)[ridx].float().cpu().numpy()
    dw = run.dweight.cpu().numpy()
    return [tol.check("y", y, y_ref, tol.bound_y(y_ref)),
            tol.check("dx", dx, dx_ref, tol.bound_dx(dx_ref, k_scale)),
            tol.check("dweight", dw, dw_ref, tol.bound_dw(dw_ref, s_scale))]


def run_all_layouts(wl, kinds=None, head_set: int = 0, rpt: int = 1, device="cuda"):
    x, dy, w = logical_inputs(wl, head_set, rpt, device)
    lays = L.workload_layouts(wl, kinds)
    runs = {k: harness.run_layout(v, x, dy, w, wl.eps, rows_per_token=rpt, device=device)
            for k, v in lays.items()}
    return x, dy, w, lays, runs

"""Bitwise batch-invariance harness.

Runs the forward and backward over every physical layout of one logical
multiset, restores the per-token outputs to logical order, and compares the
layouts bit for bit (atol = 0, rtol = 0).  Accuracy against a reference is a
separate question handled by the caller ("[WS1 Closeout][Backward] ...",
RL-Kernel #270, Acceptance criteria: invariance is bitwise after logical
aggregation, only accuracy uses a tolerance; report max abs/rel, the tensor
name and the first failing pair).  The harness also proves that the layouts
really differ (call counts, row shapes, moved rows), since comparing a layout
with itself would make every verdict a tautology ("WS1 C4 (#270) closeout
evidence", section "The matrix is falsifiable").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import layout as layout_mod

SENTINEL_BITS = 0x7FA5          # bf16 NaN pattern pre-filled into outputs: must stay in padding


@dataclass
class LayoutRun:
    name: str
    y: object                   # torch bf16 [N_tok, rpt, H], logical order
    dx: object
    dweight: object             # torch float32 [H]
    status: int
    calls: int
    rows: list
    whole_blocks: int = 0
    spill_rows: int = 0
    untouched_padding: bool = True
    h: object = None            # residual-add chain: h = bf16(x + r), logical order


@dataclass
class Diff:
    """Drift of one tensor of one layout against the reference layout: bitwise
    verdict plus the attribution metrics max / mean / p99 of |difference| and
    the first mismatching logical row ("Phase 4: single-card operator
    comparisons and drift attribution", Scope)."""
    tensor: str
    layout: str
    reference: str
    equal: bool
    mismatches: int
    max_abs: float
    max_rel: float
    first_logical_index: int
    mean_abs: float = 0.0
    p99_abs: float = 0.0


@dataclass
class InvarianceReport:
    reference: str
    diffs: list = field(default_factory=list)
    statuses: dict = field(default_factory=dict)
    distinct: dict = field(default_factory=dict)

    @property
    def green(self) -> bool:
        return (all(d.equal for d in self.diffs) and all(s == 0 for s in self.statuses.values())
                and all(self.distinct.values()))

    def first_failure(self):
        for d in self.diffs:
            if not d.equal:
                return d
        return None

    def summary(self) -> dict:
        f = self.first_failure()
        return {"green": self.green, "reference": self.reference,
                "layouts": sorted({d.layout for d in self.diffs}),
                "first_failure": None if f is None else f.__dict__,
                "statuses": self.statuses, "distinct": self.distinct}


def _bits(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16)
    if t.dtype == torch.float32:
        return t.contiguous().view(torch.int32)
    raise TypeError(t.dtype)


def bitwise_diff(name: str, a, b, layout: str, reference: str) -> Diff:
    """Compare two tensors bit for bit; NaNs compare by bit pattern."""
    import torch
    ba, bb = _bits(a).reshape(-1), _bits(b).reshape(-1)
    neq = ba != bb
    n = int(neq.sum().item())
    if n == 0:
        return Diff(name, layout, reference, True, 0, 0.0, 0.0, -1)
    fa, fb = a.reshape(-1).float(), b.reshape(-1).float()
    d = (fa - fb).abs()
    d = torch.where(torch.isnan(d), torch.full_like(d, float("inf")), d)
    rel = d / fb.abs().clamp_min(1e-30)
    first = int(torch.nonzero(neq)[0].item())
    row_len = a.reshape(a.shape[0], -1).shape[1] if a.dim() > 1 else 1
    finite = d[torch.isfinite(d)].double()
    mean = float(finite.mean().item()) if finite.numel() else float("inf")
    p99 = float(torch.quantile(finite[:1 << 24], 0.99).item()) if finite.numel() else float("inf")
    return Diff(name, layout, reference, False, n, float(d.max().item()), float(rel.max().item()),
                first // row_len, mean, p99)


def layouts_differ(ref: layout_mod.Layout, other: layout_mod.Layout) -> bool:
    """True if the physical placement differs: call count, row shapes, or a moved token."""
    if len(ref.calls) != len(other.calls) or ref.rows_per_call != other.rows_per_call:
        return True
    return any(not np.array_equal(a, b) for a, b in zip(ref.calls, other.calls))


def run_layout(lay: layout_mod.Layout, x_log, dy_log, weight, eps: float, rows_per_token: int = 1,
               device="cuda", stream=None, check_padding: bool = True) -> LayoutRun:
    """Forward + backward + dweight of one layout through the library; outputs in logical order.

    x_log, dy_log: bf16 [N_tok, rpt, H] (or [N_tok, H]) logical tensors on `device`.
    Inactive rows of the physical inputs are filled with NaN, and the outputs are
    pre-filled with a NaN sentinel that must survive in the padding.
    """
    import torch
    import invariant_rmsnorm_fwd_gb300 as rb
    H = weight.shape[0]
    R = rows_per_token
    xl = x_log.reshape(-1, R, H)
    dl = dy_log.reshape(-1, R, H)
    n_tok = xl.shape[0]
    ws = rb.DweightWorkspace(n_tok * R, H, device=device)
    y_log = torch.empty_like(xl)
    dx_log = torch.empty_like(dl)
    descs, bufs = [], []
    whole = spill = 0
    for tok in lay.calls:
        cl = rb.call_layout(tok, R, lay.n_logical_tokens, device=device)
        whole += cl.whole_blocks
        spill += cl.spill_rows
        tid = cl.tok_id.long()
        act = tid >= 0
        xp = torch.full((tok.size, R, H), float("nan"), dtype=torch.bfloat16, device=device)
        dp = torch.full_like(xp, float("nan"))
        xp[act] = xl[tid[act]]
        dp[act] = dl[tid[act]]
        yp = torch.full((tok.size, R, H), 0, dtype=torch.int16, device=device).fill_(SENTINEL_BITS).view(torch.bfloat16)
        dxp = yp.clone()
        descs.append((cl, act, tid))
        bufs.append((xp, dp, yp, dxp))
    for (cl, _, _), (xp, dp, yp, _) in zip(descs, bufs):
        rb.rmsnorm_fwd(xp, weight, cl, eps, y=yp, stream=stream)
    ws.begin(stream)
    for (cl, _, _), (xp, dp, _, dxp) in zip(descs, bufs):
        rb.rmsnorm_bwd_dx(xp, weight, dp, cl, eps, dx=dxp, workspace=ws, stream=stream)
    dw = ws.finalize(stream=stream)
    status = ws.status(stream)
    untouched = True
    for (cl, act, tid), (_, _, yp, dxp) in zip(descs, bufs):
        y_log[tid[act]] = yp[act]
        dx_log[tid[act]] = dxp[act]
        if check_padding and bool((~act).any()):
            pad = ~act
            sent = torch.tensor(SENTINEL_BITS, dtype=torch.int16, device=device)
            untouched &= bool((yp[pad].view(torch.int16) == sent).all()) and \
                bool((dxp[pad].view(torch.int16) == sent).all())
    return LayoutRun(lay.name, y_log, dx_log, dw, status, len(lay.calls), lay.rows_per_call, whole, spill,
                     untouched)


def run_layout_chain(lay: layout_mod.Layout, x_log, r_log, dy_log, dres_log, weight, eps: float, grad_scale,
                     rows_per_token: int = 1, device="cuda", stream=None) -> LayoutRun:
    """Residual add + norm forward and its backward with the loss seed's scale,
    through the library, for one layout; outputs in logical order.

    grad_scale is a float (the same 1/D for every call: the multiset's
    active-token denominator) or a callable taking a call's token ids and
    returning that call's factor (used to show that a per-call denominator is
    caught).  dweight is finalized with the float, or with 1 for a callable."""
    import torch
    import invariant_rmsnorm_fwd_gb300 as rb
    H = weight.shape[0]
    R = rows_per_token
    views = [t.reshape(-1, R, H) for t in (x_log, r_log, dy_log, dres_log)]
    n_tok = views[0].shape[0]
    ws = rb.DweightWorkspace(n_tok * R, H, device=device)
    outs = {k: torch.empty_like(views[0]) for k in ("h", "y", "dx")}
    ws.begin(stream)
    whole = spill = 0
    untouched = True
    sent = torch.tensor(SENTINEL_BITS, dtype=torch.int16, device=device)
    for tok in lay.calls:
        cl = rb.call_layout(tok, R, lay.n_logical_tokens, device=device)
        whole += cl.whole_blocks
        spill += cl.spill_rows
        tid = cl.tok_id.long()
        act = tid >= 0
        phys = []
        for v in views:
            t = torch.full((tok.size, R, H), float("nan"), dtype=torch.bfloat16, device=device)
            t[act] = v[tid[act]]
            phys.append(t)
        xp, rp, dp, drp = phys
        hp = torch.empty((tok.size, R, H), dtype=torch.int16, device=device).fill_(SENTINEL_BITS).view(torch.bfloat16)
        yp, dxp = hp.clone(), hp.clone()
        rb.rmsnorm_add_fwd(xp, rp, weight, cl, eps, h=hp, y=yp, stream=stream)
        s = grad_scale(tok) if callable(grad_scale) else grad_scale
        rb.rmsnorm_add_bwd(hp, weight, dp, cl, eps, dres=drp, grad_scale=s, dx=dxp, workspace=ws, stream=stream)
        outs["h"][tid[act]] = hp[act]
        outs["y"][tid[act]] = yp[act]
        outs["dx"][tid[act]] = dxp[act]
        if bool((~act).any()):
            pad = ~act
            untouched &= all(bool((t[pad].view(torch.int16) == sent).all()) for t in (hp, yp, dxp))
    dw = ws.finalize(stream=stream, grad_scale=1.0 if callable(grad_scale) else grad_scale)
    return LayoutRun(lay.name, outs["y"], outs["dx"], dw, ws.status(stream), len(lay.calls), lay.rows_per_call,
                     whole, spill, untouched, h=outs["h"])


def run_layout_gemm(lay: layout_mod.Layout, x_log, dy_log, device="cuda", stream=None) -> LayoutRun:
    """The linear layer's deterministic weight gradient for one layout: every call
    places its tokens, one finalize forms dW.  dW is returned as the run's
    `dweight` (FP32 [O][I]); y and dx are empty."""
    import torch
    import invariant_rmsnorm_fwd_gb300 as rb
    n_tok, I = x_log.shape
    O = dy_log.shape[1]
    ws = rb.GemmDwWorkspace(n_tok, I, O, device=device)
    ws.begin(stream)
    for tok in lay.calls:
        cl = rb.call_layout(tok, 1, lay.n_logical_tokens, device=device, with_plan=False)
        tid = cl.tok_id.long()
        act = tid >= 0
        xp = torch.full((tok.size, I), float("nan"), dtype=torch.bfloat16, device=device)
        dp = torch.full((tok.size, O), float("nan"), dtype=torch.bfloat16, device=device)
        xp[act] = x_log[tid[act]]
        dp[act] = dy_log[tid[act]]
        ws.contrib(xp, dp, cl, stream)
    dw = ws.finalize(stream=stream)
    empty = torch.empty(0, dtype=torch.bfloat16, device=device)
    return LayoutRun(lay.name, empty, empty.clone(), dw, ws.status(stream), len(lay.calls), lay.rows_per_call)


def assert_batch_invariant(runs: dict, layouts: dict, reference: str = "full") -> InvarianceReport:
    """Bitwise comparison of every layout's y, dx and dweight with the reference layout."""
    rep = InvarianceReport(reference)
    ref = runs[reference]
    for name, run in runs.items():
        rep.statuses[name] = run.status
        if name == reference:
            continue
        rep.distinct[name] = layouts_differ(layouts[reference], layouts[name])
        for t in ("y", "dx", "dweight", "h"):
            a, b = getattr(run, t), getattr(ref, t)
            if a is None and b is None:
                continue
            rep.diffs.append(bitwise_diff(t, a, b, name, reference))
    return rep

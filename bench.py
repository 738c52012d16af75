#!/usr/bin/env python3
"""Benchmark of batch-invariant RMSNorm forward + backward on GB300.

One step = the whole hot path over one batch of the workload in one physical
layout: rmsnorm_fwd on every call, rmsnorm_dweight_begin, rmsnorm_bwd_dx
(dx fused with the dweight contribution) on every call, dweight_finalize.
Inputs are resident in HBM when the timed region starts; L2 is flushed
before every timed step (a 256 MB write, then a 256 MB read so that no dirty
lines are left to be written back inside the timed region); each step is
timed with CUDA events on the launching stream.  `value` is active tokens per
second.  The default workload is c4 in its headline layout (hidden 5120,
262,144 tokens in 2^20 left-padded slots, 256 calls of 4096 slots), the
largest one that fits one GPU; the headline layouts of c1, c2 and c3 are
timed in the same run and reported under `other_workloads`.  The roofline
object reports the dominant kernel (the fused backward: its launches of one
step, timed as they run inside the step) against the measured HBM copy
bandwidth.  `e2e` is the same metric through the public API with host
buffers: plans built on the host, inputs copied in from pinned memory and y,
dx, dweight copied back, all inside the timed region.  `cpu_baseline` is the
FP64 oracle on every host core (one process per core) and on one core.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c4] [--layout L] [--also c1,c2,c3]
  python bench.py --impl reference ...   # the FP64 oracle on host cores (reported baseline)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RMSNorm fwd+bwd tokens/s and HBM GB/s (% of roofline), bitwise across layouts"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c4")
    ap.add_argument("--also", default="c1,c2,c3",
                    help="other workloads whose headline layouts are timed in the same run (comma list, '' = none)")
    ap.add_argument("--layout", default=None, help="headline layout (default: the workload's)")
    ap.add_argument("--all-layouts", action="store_true", help="also time every layout cell")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of a CUDA graph")
    ap.add_argument("--streams", type=int, default=64, help="streams the calls of a multi-call layout fork over")
    ap.add_argument("--schedule", default="lpt", choices=["lpt", "rr"],
                    help="how calls are dealt to the streams: largest first to the least-loaded stream, or round robin")
    ap.add_argument("--clock-log", default=None, help="keep the nvidia-smi clock samples in this CSV file")
    ap.add_argument("--max-tokens", type=int, default=0,
                    help="cut the workload to its first N logical tokens (profiling runs only)")
    ap.add_argument("--e2e-chunk", type=int, default=4096, help="token slots per sub-call of the e2e leg")
    ap.add_argument("--e2e-lanes", type=int, default=1, help="copy streams per direction in the e2e leg")
    ap.add_argument("--e2e-first", type=int, default=2048,
                    help="token slots of the first e2e sub-call (doubling up to --e2e-chunk)")
    ap.add_argument("--gemm", action="store_true",
                    help="the linear layer's deterministic weight gradient (in = out = hidden) instead of the norm")
    ap.add_argument("--chain", action="store_true",
                    help="residual add + norm forward and its backward with the residual gradient and the "
                         "loss seed's 1/D (D = active tokens of the multiset); no e2e or CPU legs")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def source_sha256():
    """Hash of the library sources, to tell whether a recorded ncu traffic still applies."""
    import glob
    import hashlib
    files = sorted(glob.glob(os.path.join(ROOT, "invariant_rmsnorm_fwd_gb300", "csrc", "*")))
    files += sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()


def recorded_traffic(config: str, layout: str):
    """DRAM bytes of the backward phase (the sum over its launches) from
    profiles/traffic.json, or None if no record is for this workload and layout
    or the kernels changed since the record was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    sha = source_sha256()
    for rec in d.get("records", [d]):
        if rec.get("workload") == config and rec.get("layout") == layout and rec.get("source_sha256") == sha:
            return int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])
    return None


def workload_desc(wl, lay_name, n_phys):
    heads = "x".join(str(h) for h in wl.heads)
    return (f"{wl.name}: hidden={wl.hidden}, heads={heads}, {len(wl.lengths)} samples, "
            f"{wl.n_tokens} active tokens, layout={lay_name} ({n_phys} physical token slots)")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path=None):
        """Samples go to `path` (the --clock-log option) or to a temporary file."""
        import tempfile
        self.proc = None
        self.gpu = gpu_index
        self.tmp = not path
        if path:
            self.path = path
        else:
            fd, self.path = tempfile.mkstemp(prefix=f"clocks_gpu{gpu_index}_", suffix=".csv")
            os.close(fd)

    def start(self):
        """Start sampling every 100 ms; returns once the first sample is on disk (or after 5 s)."""
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            if self.tmp and os.path.exists(self.path):
                os.unlink(self.path)
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if self.tmp:
            os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm

class L2Flush:
    """Runs between timed steps, untimed: writes a 256 MB buffer (twice the 129 MB L2),
    then reads a second 256 MB buffer so that the dirty lines of the write are written
    back before the timed region instead of during it.  L2 ends clean and holds none
    of the workload's data."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        self.r = torch.ones(64 << 20, dtype=torch.int32, device=device)
        self.sink = torch.empty((), dtype=torch.int32, device=device)

    def __call__(self):
        import torch
        self.w.fill_(1)
        torch.amax(self.r, dim=0, out=self.sink)


class Call:
    """Physical buffers of one call: x, dy, y, dx (and r, dres, h for the chain)."""

    def __init__(self, cl, xp, dp, yp, dxp, rp=None, drp=None, hp=None):
        self.cl, self.xp, self.dp, self.yp, self.dxp = cl, xp, dp, yp, dxp
        self.rp, self.drp, self.hp = rp, drp, hp


class Step:
    """Device-resident buffers of one layout and the launch sequence of one step.
    With `chain`, the step is the residual add + norm forward and the backward
    with the residual gradient, scaled by the loss seed's 1/D."""

    def __init__(self, wl, lay, x_log, dy_log, w, rpt, device, r_log=None, dres_log=None, n_streams=64,
                 schedule="lpt"):
        import torch
        import invariant_rmsnorm_fwd_gb300 as rb
        self.rb = rb
        H = wl.hidden
        self.H, self.rpt, self.eps = H, rpt, wl.eps
        self.w = w
        self.chain = r_log is not None
        self.scale = 1.0 / wl.n_tokens if self.chain else None
        self.calls = []
        for tok in lay.calls:
            cl = rb.call_layout(tok, rpt, lay.n_logical_tokens, device=device)
            tid = cl.tok_id.long()
            act = tid >= 0

            def place(src):
                t = torch.zeros((tok.size, rpt, H), dtype=torch.bfloat16, device=device)
                t[act] = src[tid[act]]
                return t
            xp, dp = place(x_log), place(dy_log)
            if self.chain:
                self.calls.append(Call(cl, xp, dp, torch.empty_like(xp), torch.empty_like(xp), place(r_log),
                                       place(dres_log), torch.empty_like(xp)))
            else:
                self.calls.append(Call(cl, xp, dp, torch.empty_like(xp), torch.empty_like(xp)))
        self.ws = rb.DweightWorkspace(wl.n_tokens * rpt, H, device=device)
        self.dw = torch.empty(H, dtype=torch.float32, device=device)
        self.n_active = wl.n_tokens
        self.n_streams = n_streams
        self.schedule = schedule
        self.bwd_events = []

    def fwd_call(self, c, st):
        if self.chain:
            self.rb.rmsnorm_add_fwd(c.xp, c.rp, self.w, c.cl, self.eps, h=c.hp, y=c.yp, stream=st)
        else:
            self.rb.rmsnorm_fwd(c.xp, self.w, c.cl, self.eps, y=c.yp, stream=st)

    def bwd_call(self, c, st):
        if self.chain:
            self.rb.rmsnorm_add_bwd(c.hp, self.w, c.dp, c.cl, self.eps, dres=c.drp, grad_scale=self.scale,
                                    dx=c.dxp, workspace=self.ws, stream=st)
        else:
            self.rb.rmsnorm_bwd_dx(c.xp, self.w, c.dp, c.cl, self.eps, dx=c.dxp, workspace=self.ws, stream=st)

    def finalize(self, st):
        self.ws.finalize(self.dw, st, grad_scale=self.scale)

    def _assignment(self, n_lanes):
        """(call index, lane) pairs in issue order.  Calls without active tokens
        launch nothing and are left out; with schedule "lpt" the others go, largest
        first, to the lane with the fewest active rows so far (longest processing
        time first), so the lanes end close together; "rr" deals them round robin
        in layout order."""
        sizes = [int((c.cl.tok_id >= 0).sum().item()) if c.cl.n_tokens else 0 for c in self.calls]
        idx = [i for i, n in enumerate(sizes) if n > 0]
        if self.schedule == "rr":
            return [(i, k % n_lanes) for k, i in enumerate(idx)]
        load = [0] * n_lanes
        out = []
        for i in sorted(idx, key=lambda i: -sizes[i]):
            lane = min(range(n_lanes), key=lambda j: load[j])
            load[lane] += sizes[i]
            out.append((i, lane))
        return out

    def _fan(self, fn, stream):
        """Calls of a multi-call layout are independent (they touch disjoint rows and
        blocks of the workspace), so they are spread over n_streams streams (64 by default) that
        fork from and join back into `stream`; one-call layouts stay on `stream`."""
        import torch
        lanes = self._lanes(stream)
        if len(lanes) == 1:
            for c in self.calls:
                fn(c, stream)
            return
        if getattr(self, "_plan", None) is None:
            self._plan = self._assignment(len(lanes))
        ev = torch.cuda.Event()
        ev.record(stream)
        used = sorted({lane for _, lane in self._plan})
        for lane in used:
            lanes[lane].wait_event(ev)
        for i, lane in self._plan:
            fn(self.calls[i], lanes[lane])
        for lane in used:
            e = torch.cuda.Event()
            e.record(lanes[lane])
            stream.wait_event(e)

    def run(self, stream):
        self._fan(self.fwd_call, stream)
        self.ws.begin(stream)
        self._fan(self.bwd_call, stream)
        self.finalize(stream)

    def bwd_phase(self, stream):
        """The backward launches of one step alone (the workspace begun beforehand)."""
        self._fan(self.bwd_call, stream)

    def fwd_phase(self, stream):
        """The forward launches of one step alone."""
        self._fan(self.fwd_call, stream)

    def fin_phase(self, stream):
        """The finalize of one step alone (over the workspace of the last backward)."""
        self.finalize(stream)

    def _lanes(self, stream):
        import torch
        if len(self.calls) == 1:
            return [stream]
        if getattr(self, "_side", None) is None:
            self._side = [torch.cuda.Stream(device=self.dw.device) for _ in range(self.n_streams)]
        return self._side

    def gather(self, n_tok):
        import torch
        y = torch.empty((n_tok, self.rpt, self.H), dtype=torch.bfloat16, device=self.dw.device)
        dx = torch.empty_like(y)
        h = torch.empty_like(y) if self.chain else None
        for c in self.calls:
            tid = c.cl.tok_id.long()
            act = tid >= 0
            y[tid[act]] = c.yp[act]
            dx[tid[act]] = c.dxp[act]
            if self.chain:
                h[tid[act]] = c.hp[act]
        return (y, dx, self.dw.clone()) + ((h,) if self.chain else ())


def time_steps(step, stream, steps, warmup, flush, dist=None, graph=True):
    """W eager warm-up steps, then K timed steps (CUDA-graph replays of one whole
    step when graph=True), each preceded by an untimed L2 flush; returns ms per step."""
    import torch
    for _ in range(warmup):
        step.run(stream)
    torch.cuda.synchronize()
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            step.run(torch.cuda.current_stream())
        torch.cuda.synchronize()
        g.replay()                               # one untimed replay
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if g is not None:
            g.replay()
        else:
            step.run(stream)
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return [a.elapsed_time(b) for a, b in times], g


def time_bwd_kernel(step_objs, stream, reps, flush):
    """Duration of each fused-backward launch (CUDA events on the launching stream)."""
    import torch
    per = []
    for _ in range(reps):
        for so in step_objs:
            so.ws.begin(stream)
            for c in so.calls:
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                so.bwd_call(c, stream)
                e1.record(stream)
                per.append((e0, e1))
            so.finalize(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in per]


def time_phase(multi, stream, reps, flush, which="bwd"):
    """Duration of one phase of a step as it runs inside the step: every forward
    ("fwd") or fused-backward ("bwd") launch of every normed tensor (all calls
    of a many-call layout, forked over the step's streams), or the finalize
    ("fin") of each workspace over what the last backward left in it,
    captured as one CUDA graph and replayed between two CUDA events on the
    launching stream.  For the backward each workspace is begun (eagerly,
    outside the events); L2 is flushed before each replay."""
    import torch
    phase = {"bwd": multi.bwd_phase, "fwd": multi.fwd_phase, "fin": multi.fin_phase}[which]

    def prep():
        if which == "bwd":
            for s in multi.steps:
                s.ws.begin(stream)
    prep()
    phase(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.graph(g, stream=cap):
        phase(torch.cuda.current_stream())
    torch.cuda.synchronize()
    evs = []
    for _ in range(reps):
        prep()
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    if which == "bwd":
        for s in multi.steps:
            s.finalize(stream)
        torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def e2e_subcalls(lay, chunk_tokens, first_tokens):
    """Token slots of the sub-calls the end-to-end leg issues, in order.  Every call
    of the layout is cut into pieces of at most `chunk_tokens` slots, the first
    pieces growing from `first_tokens` (doubling) so that compute starts after a
    short first copy; padding slots at either end of a piece are dropped (their
    rows are neither read nor written by the kernels) and all-padding pieces are
    skipped.  The outputs do not depend on this cut."""
    subs = []
    size = min(first_tokens or chunk_tokens, chunk_tokens)
    for tok in lay.calls:
        i = 0
        while i < tok.size:
            t = tok[i:i + size]
            i += size
            size = min(size * 2, chunk_tokens)
            act = np.nonzero(t >= 0)[0]
            if act.size:
                subs.append(np.ascontiguousarray(t[act[0]:act[-1] + 1], dtype=np.int32))
    return subs


def e2e_steps(wl, lay, norms, steps, warmup, device, chunk_tokens=4096, copy_lanes=1, first_tokens=2048):
    """Public API with host buffers.  `norms` lists the normed tensors of one step as
    (rows_per_token, x, dy, weight) with x and dy in logical order on the host (Q
    and K of a per-head norm are two).  Per step, for every sub-call (see
    e2e_subcalls) of every tensor, in one pipeline: copy x and dy in from pinned
    memory, build the plan on the host while they copy, copy token ids and plan
    in, run forward and fused backward, copy y and dx back; then finalize each
    dweight and copy it back.  Copy-in streams, the compute stream and copy-out
    streams (`copy_lanes` of each) overlap.  Returns (ms per step, h2d bytes, d2h
    bytes, description, per tensor (y, dx, dweight) of the last step gathered to
    logical order on the host)."""
    import torch
    import invariant_rmsnorm_fwd_gb300 as rb
    H = wl.hidden
    comp = torch.cuda.current_stream()
    s_ins = [torch.cuda.Stream(device=device) for _ in range(copy_lanes)]
    s_outs = [torch.cuda.Stream(device=device) for _ in range(copy_lanes)]
    cuts = e2e_subcalls(lay, chunk_tokens, first_tokens)
    subs = []                                   # (tensor index, token slots), tensors interleaved
    for tok in cuts:
        for n in range(len(norms)):
            subs.append((n, tok))
    # the caller's pinned host data, laid out physically per sub-call
    host, dev, meta_h, meta_d = [], [], [], []
    for n, tok in subs:
        rpt, x_log_host, dy_log_host, _ = norms[n]
        act = tok >= 0
        xh = torch.zeros((tok.size, rpt, H), dtype=torch.bfloat16).pin_memory()
        dh = torch.zeros_like(xh).pin_memory()
        idx = torch.as_tensor(tok[act]).long()
        xh[torch.as_tensor(act)] = x_log_host[idx]
        dh[torch.as_tensor(act)] = dy_log_host[idx]
        host.append((xh, dh, torch.empty_like(xh).pin_memory(), torch.empty_like(xh).pin_memory()))
        dev.append(tuple(torch.empty(xh.shape, dtype=torch.bfloat16, device=device) for _ in range(4)))
        cap = rb.plan_capacity(tok.size, rpt)
        meta_h.append((torch.empty(tok.size, dtype=torch.int32).pin_memory(),
                       torch.empty(cap, dtype=torch.uint8).pin_memory()))
        meta_d.append((torch.empty(tok.size, dtype=torch.int32, device=device),
                       torch.empty(cap, dtype=torch.uint8, device=device)))
    wss = [rb.DweightWorkspace(wl.n_tokens * rpt, H, device=device) for rpt, _, _, _ in norms]
    dw_d = [torch.empty(H, dtype=torch.float32, device=device) for _ in norms]
    dw_h = [torch.empty(H, dtype=torch.float32).pin_memory() for _ in norms]
    counts = {}

    def one():
        h2d = d2h = 0
        for ws in wss:
            ws.begin(comp)
        for i, ((n, tok), (th, ph), (td, pd), (xh, dh, yh, dxh), (xd, dd, yd, dxd)) in enumerate(
                zip(subs, meta_h, meta_d, host, dev)):
            rpt, _, _, w = norms[n]
            s_in, s_out = s_ins[i % copy_lanes], s_outs[i % copy_lanes]
            with torch.cuda.stream(s_in):
                # the bulk copies go first: the host builds this sub-call's plan while they run
                xd.copy_(xh, non_blocking=True)
                dd.copy_(dh, non_blocking=True)
                pbytes, items, whole, spill = rb.plan_build(tok, rpt, lay.n_logical_tokens, out=ph.numpy())
                th.numpy()[:] = tok
                td.copy_(th, non_blocking=True)
                pd[:pbytes.size].copy_(ph[:pbytes.size], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            h2d += xh.numel() * 2 * 2 + tok.nbytes + pbytes.size
            cl = rb.CallLayout(td, pd, items, tok.size, rpt, lay.n_logical_tokens, whole, spill)
            comp.wait_event(ready)
            rb.rmsnorm_fwd(xd, w, cl, wl.eps, y=yd, stream=comp)
            e1 = torch.cuda.Event()
            e1.record(comp)                        # y can leave while the backward runs
            rb.rmsnorm_bwd_dx(xd, w, dd, cl, wl.eps, dx=dxd, workspace=wss[n], stream=comp)
            e2 = torch.cuda.Event()
            e2.record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e1)
                yh.copy_(yd, non_blocking=True)
                s_out.wait_event(e2)
                dxh.copy_(dxd, non_blocking=True)
            d2h += yd.numel() * 2 * 2
        for ws, dd_, dh_ in zip(wss, dw_d, dw_h):
            ws.finalize(dd_, comp)
            fin = torch.cuda.Event()
            fin.record(comp)
            with torch.cuda.stream(s_outs[0]):
                s_outs[0].wait_event(fin)
                dh_.copy_(dd_, non_blocking=True)
            d2h += H * 4
        torch.cuda.synchronize()
        counts["h2d"], counts["d2h"] = h2d, d2h

    for _ in range(warmup):
        one()
    ts = []
    for _ in range(steps):
        t0 = time.perf_counter()
        one()
        ts.append((time.perf_counter() - t0) * 1e3)
    outs = []
    for n, (rpt, _, _, _) in enumerate(norms):
        y = torch.zeros((wl.n_tokens, rpt, H), dtype=torch.bfloat16)
        dx = torch.zeros_like(y)
        for (m, tok), (_, _, yh, dxh) in zip(subs, host):
            if m == n:
                act = torch.as_tensor(tok >= 0)
                idx = torch.as_tensor(tok[tok >= 0]).long()
                y[idx] = yh[act]
                dx[idx] = dxh[act]
        outs.append((y, dx, dw_h[n].clone()))
    sizes = sorted({int(t.size) for t in cuts})
    desc = (f"{len(subs)} sub-calls ({len(cuts)} per normed tensor, token slots from {sizes[0]} to {sizes[-1]}: "
            f"the first ones ramp up from {first_tokens}, at most {chunk_tokens}, padding at their ends not "
            f"copied), pipelined over {copy_lanes} copy-in streams, the compute stream and {copy_lanes} "
            f"copy-out streams; every plan built on the host each step while its sub-call's inputs copy")
    return statistics.median(ts), counts["h2d"], counts["d2h"], desc, outs


def _oracle_rows(x, dy, w, eps, seconds):
    """Runs the oracle's forward and backward over the rows x, dy (uint16 bf16
    patterns [n, H]) again and again for about `seconds`; returns (rows done, s)."""
    import oracle
    n = x.shape[0]
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle.forward(x, w, eps)
        oracle.backward(x, w, dy, eps)
        done += n
    return done, time.perf_counter() - t0


def _oracle_worker(job):
    x, dy, w, eps, seconds = job
    return _oracle_rows(x, dy, w, eps, seconds)


def cpu_baseline(wl, x_log, dy_log, w, seconds):
    """The FP64 oracle as it stands (plain single-threaded C) on a bounded sample of
    rows: once on one core, then as one process per host core (spawned, each with
    its own slice of the sample rows, all running at once).  Returns the all-core
    figure with the one-core figure beside it."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import torch
    H = wl.hidden
    to_u16 = lambda t: t.reshape(-1, H).contiguous().view(torch.int16).numpy().view(np.uint16)
    xr, dr = to_u16(x_log), to_u16(dy_log)
    wu = w.contiguous().view(torch.int16).numpy().view(np.uint16)
    n = xr.shape[0]
    rows_per_token = sum(wl.heads)              # every normed tensor of a token (Q and K heads)
    chunk = max(1, min(n, (1 << 22) // H))
    done1, dt1 = _oracle_rows(xr[:chunk], dr[:chunk], wu, wl.eps, seconds)
    one = done1 / rows_per_token / dt1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    per = max(1, n // cores)
    jobs = [(xr[i * per:(i + 1) * per], dr[i * per:(i + 1) * per], wu, wl.eps, seconds) for i in range(cores)]
    with cf.ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
        res = list(ex.map(_oracle_worker, jobs))
    done_all = sum(r[0] for r in res)
    dt_all = max(r[1] for r in res)
    allc = done_all / rows_per_token / dt_all
    return {"value": allc, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "one_core": {"value": one, "unit": "tokens/s", "cores": 1,
                         "sample": f"{done1} logical rows (the first {chunk}, cycled) in {dt1:.1f} s"},
            "sample": f"{n} logical rows of hidden {H} (the workload's first rows), fwd + bwd incl. dweight "
                      f"in the FP64 C oracle (single-threaded code, unchanged): one spawned process per "
                      f"host core ({cores}), each cycling its own slice of {per} rows for ~{seconds:.0f} s, "
                      f"{done_all} rows in all; rate = rows / slowest process's time; a token is "
                      f"{rows_per_token} such rows"}


class Multi:
    """The normed tensors of one step (Q and K of a per-head norm) are
    independent ops with their own weights and workspaces: they fork onto
    their own streams and join back, as a model issues them."""

    def __init__(self, steps, device):
        import torch
        self.steps = steps
        self.side = [torch.cuda.Stream(device=device) for _ in steps[1:]]

    def _fork(self, stream, fn):
        import torch
        if len(self.steps) == 1:
            fn(self.steps[0], stream)
            return
        ev = torch.cuda.Event()
        ev.record(stream)
        for st, s in zip(self.side, self.steps[1:]):
            st.wait_event(ev)
            fn(s, st)
        fn(self.steps[0], stream)
        for st in self.side:
            e = torch.cuda.Event()
            e.record(st)
            stream.wait_event(e)

    def run(self, stream):
        self._fork(stream, lambda s, st: s.run(st))

    def bwd_phase(self, stream):
        self._fork(stream, lambda s, st: s.bwd_phase(st))

    def fwd_phase(self, stream):
        self._fork(stream, lambda s, st: s.fwd_phase(st))

    def fin_phase(self, stream):
        self._fork(stream, lambda s, st: s.fin_phase(st))


def workload_data(wl, device, chain=False):
    """Logical inputs of every normed tensor of a workload: (rows per token, x, dy, w[, r, dres])."""
    import synth
    out = []
    for hs, rpt in enumerate(wl.heads):
        n_rows = wl.n_tokens * rpt
        shape = (wl.n_tokens, rpt, wl.hidden)
        x = synth.logical_tensor(wl, synth.TAG_X, n_rows, wl.x_std, hs, device=device).reshape(shape)
        dy = synth.logical_tensor(wl, synth.TAG_DY, n_rows, wl.dy_std, hs, device=device).reshape(shape)
        w = synth.weight(wl, hs, device=device)
        extra = ()
        if chain:
            r = synth.logical_tensor(wl, synth.TAG_RES, n_rows, wl.x_std, hs, device=device)
            dres = synth.logical_tensor(wl, synth.TAG_DRES, n_rows, wl.dy_std, hs, device=device)
            extra = (r.reshape(shape), dres.reshape(shape))
        out.append((rpt, x, dy, w) + extra)
    return out


def measure(wl, lay, data, args, device, flush, stream, hbm_peak, dist=None, sample_clocks=None):
    """Times one workload in one layout: whole steps (CUDA-graph replays), the
    backward phase inside the step, each backward launch alone and the forward
    alone.  Returns (dict of figures, the Multi of steps)."""
    import torch
    import invariant_rmsnorm_fwd_gb300 as rb
    steps = [Step(wl, lay, d[1], d[2], d[3], d[0], device, *d[4:], n_streams=args.streams,
                  schedule=args.schedule) for d in data]
    multi = Multi(steps, device)
    multi.run(stream)                           # kernels of one step, counted on an eager step
    torch.cuda.synchronize()
    l0 = rb.kernel_launches()
    multi.run(stream)
    torch.cuda.synchronize()
    launches = rb.kernel_launches() - l0
    if sample_clocks is not None:
        sample_clocks.start()
    ms, graph = time_steps(multi, stream, args.steps, args.warmup, flush, dist, graph=not args.no_graph)
    clk = None
    if sample_clocks is not None:
        # keep the same step running (untimed) so the clock samples cover the load
        t_end = time.time() + 0.6
        while time.time() < t_end:
            for _ in range(20):
                if graph is not None:
                    graph.replay()
                else:
                    multi.run(stream)
            torch.cuda.synchronize()
        clk = sample_clocks.stop()
    ms_step = statistics.mean(ms)
    if dist is not None:
        t = torch.tensor([ms_step], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_step = float(t.item())
    reps = max(3, args.steps // 2)
    phase_ms = statistics.mean(time_phase(multi, stream, reps, flush, "bwd"))
    bwd_ms = time_bwd_kernel(steps, stream, 1 if len(lay.calls) > 16 else reps, flush)
    fwd_ms = time_phase(multi, stream, reps, flush, "fwd")
    fin_ms = time_phase(multi, stream, reps, flush, "fin")
    heff = wl.hidden * sum(wl.heads)
    n_act = wl.n_tokens
    fwd_b, bwd_b = (8.0, 8.0) if args.chain else (4.0, 6.0)
    alg_step = (fwd_b + bwd_b) * heff * n_act
    alg_bwd = bwd_b * heff * n_act
    bwd_launches = len(lay.calls) * len(wl.heads)
    iso_ms = statistics.mean(bwd_ms)
    r = {"ms_step": ms_step, "launches": int(launches), "clocks": clk, "graph": graph is not None,
         "tokens_per_s": n_act / (ms_step * 1e-3),
         "hbm_gbs_step": alg_step / (ms_step * 1e-3) / 1e9,
         "frac_step": alg_step / (ms_step * 1e-3) / 1e9 / hbm_peak,
         "bwd_phase_ms": phase_ms, "bwd_alg_bytes": alg_bwd, "bwd_launches": bwd_launches,
         "bwd_gbs": alg_bwd / (phase_ms * 1e-3) / 1e9,
         "bwd_iso_launch_ms": iso_ms, "bwd_iso_gbs": alg_bwd / bwd_launches / (iso_ms * 1e-3) / 1e9,
         "fwd_gbs": fwd_b * heff * n_act / (statistics.mean(fwd_ms) * 1e-3) / 1e9,
         "fin_phase_ms": statistics.mean(fin_ms)}
    return r, multi


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if args.gemm:
        return gemm_bench(args, rank, world)

    import torch
    import synth
    from invariant_rmsnorm_fwd_gb300 import layout as L, harness

    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist = tdist

    wl = synth.config(args.config)
    if args.max_tokens:
        wl = synth.truncated(wl, args.max_tokens)
    lay_name = args.layout or wl.headline
    rpt_list = list(wl.heads)
    hbm_peak, peak_kind = measured_peaks()
    flush = L2Flush(device)
    stream = torch.cuda.current_stream()

    steps_data = workload_data(wl, device, args.chain)
    lay = L.workload_layouts(wl, kinds=[lay_name])[lay_name]
    m, multi = measure(wl, lay, steps_data, args, device, flush, stream, hbm_peak, dist,
                       ClockSampler(local, args.clock_log))
    step_objs = multi.steps
    ms_step = m["ms_step"]
    H = wl.hidden
    n_act = wl.n_tokens
    bwd_calls = m["bwd_launches"]
    traffic = recorded_traffic(args.config, lay_name) if not args.chain and not args.max_tokens else None
    kernel = ("residual-add backward (dh + dweight leaves), rmsnorm_add_bwd" if args.chain
              else "fused backward (dx + dweight leaves), rmsnorm_bwd_dx")

    line = {
        "metric": METRIC,
        "value": round(n_act / (ms_step * 1e-3) * world, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "io_dtype": "bf16",
        "data": "synthetic (seeded SplitMix64/Box-Muller, keyed by logical token id)",
        "config": {"workload": workload_desc(wl, lay_name, lay.n_physical), "hidden": H,
                   "heads": list(wl.heads), "tokens": n_act, "layout": lay_name, "calls": len(lay.calls),
                   "l2": "flushed before every timed step (256 MB write, then a 256 MB read so no dirty lines remain); inputs already in HBM",
                   "launch": "one CUDA graph replay per step" if m["graph"] else "eager launches",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "hbm_gbs_step": round(m["hbm_gbs_step"], 1),
        "frac_step": round(m["frac_step"], 4),
        "fwd_gbs": round(m["fwd_gbs"], 1),
        "fin_phase_ms": round(m["fin_phase_ms"], 5),
        "roofline": {"bound": "hbm", "kernel": kernel,
                     "achieved": round(m["bwd_gbs"], 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(m["bwd_gbs"] / hbm_peak, 4),
                     "traffic": traffic,
                     "peak_source": peak_kind,
                     "algorithmic_bytes": m["bwd_alg_bytes"],
                     "launches": bwd_calls,
                     "launch_ms": round(m["bwd_phase_ms"], 5),
                     "timing": ("the backward phase of the step: all its launches (forked over the step's "
                                "streams when a layout has several calls), one CUDA-graph replay between "
                                "CUDA events on the launching stream, L2 flushed before; achieved = "
                                "algorithmic_bytes / launch_ms"),
                     "isolated_launch": {"ms": round(m["bwd_iso_launch_ms"], 5),
                                         "gbs": round(m["bwd_iso_gbs"], 1),
                                         "how": "each launch alone after an L2 flush, mean over launches"}},
        "gpu_launches": m["launches"] * args.steps,
        "gpu_launches_per_step": m["launches"],
        "clocks": m["clocks"],
    }

    if rank == 0 and args.all_layouts:
        per = {}
        ref_out = None
        bitwise = True
        for k, v in L.workload_layouts(wl).items():
            so = [Step(wl, v, d[1], d[2], d[3], d[0], device, *d[4:], n_streams=args.streams,
                       schedule=args.schedule) for d in steps_data]
            mm = Multi(so, device)
            t, _ = time_steps(mm, stream, max(3, args.steps // 2), 2, flush, graph=not args.no_graph)
            per[k] = {"ms": round(statistics.mean(t), 4), "calls": len(v.calls),
                      "tokens_per_s": round(n_act / (statistics.mean(t) * 1e-3), 1)}
            outs = [s.gather(wl.n_tokens) for s in so]
            if ref_out is None:
                ref_out = outs
            else:
                for a, b in zip(outs, ref_out):
                    for ta, tb in zip(a, b):
                        bitwise &= harness.bitwise_diff("t", ta, tb, k, "ref").equal
            del so, mm
        line["layouts"] = per
        line["bitwise_across_layouts"] = bool(bitwise)

    if args.chain:
        line["config"]["chain"] = ("h = bf16(x + r), y = RMSNorm(h); dh = bf16(dx/D + dres), dweight/D; "
                                   "D = active tokens of the multiset")
    if rank == 0 and not args.no_e2e and not args.chain:
        norms = [(d[0], d[1].cpu(), d[2].cpu(), d[3]) for d in steps_data]
        tot_ms, tot_in, tot_out, desc, e2e_out = e2e_steps(wl, lay, norms, max(10, args.steps), 3, device,
                                                           args.e2e_chunk, args.e2e_lanes, args.e2e_first)
        # the host-buffer path must give the device path's outputs bit for bit
        e2e_bitwise = True
        for s_obj, got in zip(step_objs, e2e_out):
            for a, b in zip(s_obj.gather(wl.n_tokens), got):
                e2e_bitwise &= harness.bitwise_diff("t", a.cpu(), b, "e2e", "device").equal
        line["e2e"] = {"value": round(n_act / (tot_ms * 1e-3) * world, 1), "unit": "tokens/s",
                       "h2d_bytes_per_step": int(tot_in), "d2h_bytes_per_step": int(tot_out),
                       "ms_per_step": round(tot_ms, 3), "pipeline": desc, "bitwise_vs_device_path": bool(e2e_bitwise),
                       "link_gbs": round((tot_in + tot_out) / (tot_ms * 1e-3) / 1e9, 1)}
        del norms, e2e_out

    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.chain:
        _, x, dy, w = steps_data[0][:4]
        n_cpu = min(x.shape[0], 4096)
        line["cpu_baseline"] = cpu_baseline(wl, x[:n_cpu].cpu(), dy[:n_cpu].cpu(), w.cpu(), args.cpu_seconds)

    # the other workloads' headline layouts, measured in the same run (step and backward phase)
    others = [c for c in (args.also.split(",") if args.also else []) if c and c != args.config]
    if others and not args.max_tokens:
        del multi, step_objs, steps_data
        torch.cuda.empty_cache()
        per_cfg = {}
        for c in others:
            wlc = synth.config(c)
            layc = L.workload_layouts(wlc, kinds=[wlc.headline])[wlc.headline]
            data = workload_data(wlc, device, args.chain)
            mc, mm = measure(wlc, layc, data, args, device, flush, stream, hbm_peak, dist)
            per_cfg[c] = {"workload": workload_desc(wlc, wlc.headline, layc.n_physical),
                          "ms_per_step": round(mc["ms_step"], 4), "tokens_per_s": round(mc["tokens_per_s"], 1),
                          "hbm_gbs_step": round(mc["hbm_gbs_step"], 1), "frac_step": round(mc["frac_step"], 4),
                          "bwd_phase_ms": round(mc["bwd_phase_ms"], 5), "bwd_gbs": round(mc["bwd_gbs"], 1),
                          "bwd_frac": round(mc["bwd_gbs"] / hbm_peak, 4), "bwd_launches": mc["bwd_launches"],
                          "fwd_gbs": round(mc["fwd_gbs"], 1), "fin_phase_ms": round(mc["fin_phase_ms"], 5),
                          "gpu_launches_per_step": mc["launches"]}
            del mm, data
            torch.cuda.empty_cache()
        line["other_workloads"] = per_cfg
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def gemm_bench(args, rank, world):
    """The deterministic weight gradient of a linear layer y = x W^T with in =
    out = hidden, over the workload's tokens in its headline layout: per step
    begin, one placement call per layout call, one finalize (the GEMM)."""
    import torch
    import synth
    import invariant_rmsnorm_fwd_gb300 as rb
    from invariant_rmsnorm_fwd_gb300 import layout as L
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    wl = synth.config(args.config)
    if args.max_tokens:
        wl = synth.truncated(wl, args.max_tokens)
    lay_name = args.layout or wl.headline
    lay = L.workload_layouts(wl, kinds=[lay_name])[lay_name]
    H, n = wl.hidden, wl.n_tokens
    x = synth.logical_tensor(wl, synth.TAG_X, n, wl.x_std, device=device)
    dy = synth.logical_tensor(wl, synth.TAG_DY, n, wl.dy_std, device=device)
    calls = []
    for tok in lay.calls:
        cl = rb.call_layout(tok, 1, lay.n_logical_tokens, device=device, with_plan=False)
        tid = cl.tok_id.long()
        act = tid >= 0
        xp = torch.zeros((tok.size, H), dtype=torch.bfloat16, device=device)
        dp = torch.zeros_like(xp)
        xp[act] = x[tid[act]]
        dp[act] = dy[tid[act]]
        calls.append((cl, xp, dp))
    ws = rb.GemmDwWorkspace(n, H, H, device=device)
    dw = torch.empty(H, H, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()

    class G:
        def run(self, st):
            ws.begin(st)
            for cl, xp, dp in calls:
                ws.contrib(xp, dp, cl, st)
            ws.finalize(dw, stream=st)

    g = G()
    flush = L2Flush(device)
    g.run(stream)
    torch.cuda.synchronize()
    l0 = rb.kernel_launches()
    g.run(stream)
    torch.cuda.synchronize()
    launches = rb.kernel_launches() - l0
    clocks = ClockSampler(local, args.clock_log)
    clocks.start()
    ms, graph = time_steps(g, stream, args.steps, args.warmup, flush, None, graph=not args.no_graph)
    clk = clocks.stop()
    # the finalize alone (flag check + GEMM), CUDA events on its stream
    fin = []
    for _ in range(max(3, args.steps // 2)):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ws.finalize(dw, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        fin.append(e0.elapsed_time(e1))
    fin_ms = statistics.median(fin)
    ms_step = statistics.mean(ms)
    flops = 2.0 * n * H * H
    peak_tf, peak_src = 1900.0, "fallback (bf16 dense burst)"
    try:
        mp = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak_tf, peak_src = float(mp["bf16_tflops"]), "measured (cuBLAS bf16 GEMM burst)"
    except Exception:
        pass
    line = {
        "metric": "linear-layer weight gradient (det_gemm dW) tokens/s, bitwise across layouts",
        "value": round(n / (ms_step * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 accumulate", "io_dtype": "bf16",
        "data": "synthetic (seeded SplitMix64/Box-Muller, keyed by logical token id)",
        "config": {"workload": workload_desc(wl, lay_name, lay.n_physical) + f", linear {H} -> {H}",
                   "calls": len(lay.calls), "l2": "flushed before every timed step",
                   "launch": "one CUDA graph replay per step" if graph is not None else "eager launches"},
        "roofline": {"bound": "tensor", "kernel": "finalize (flag check + tcgen05 GEMM, FP32 accumulate in tensor memory)",
                     "achieved": round(flops / (fin_ms * 1e-3) / 1e12, 1), "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(flops / (fin_ms * 1e-3) / 1e12 / peak_tf, 4), "traffic": None,
                     "peak_source": peak_src, "launch_ms": round(fin_ms, 5)},
        "placement_gbs": round(4.0 * H * n * 2 / ((ms_step - fin_ms) * 1e-3) / 1e9, 1),
        "gpu_launches": int(launches) * args.steps, "gpu_launches_per_step": int(launches),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def reference_arm(args, rank, world):
    """The oracle (FP64 C, as it stands) on every host core: one spawned process
    per core, each running the oracle over its own slice of a bounded sample of
    the workload's rows for a fixed time per step."""
    if rank != 0:
        return
    import concurrent.futures as cf
    import multiprocessing as mp
    import torch
    import synth
    from invariant_rmsnorm_fwd_gb300 import layout as L
    wl = synth.config(args.config)
    lay_name = args.layout or wl.headline
    lay = L.workload_layouts(wl, kinds=[lay_name])[lay_name]
    rpt = wl.heads[0]
    H = wl.hidden
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    per_core = max(8, (1 << 21) // H)
    n_rows = min(wl.n_tokens * rpt, per_core * cores)
    to_u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    x = to_u16(synth.logical_tensor(wl, synth.TAG_X, n_rows, wl.x_std, 0))
    dy = to_u16(synth.logical_tensor(wl, synth.TAG_DY, n_rows, wl.dy_std, 0))
    w = to_u16(synth.weight(wl, 0))
    per = max(1, n_rows // cores)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    rows_per_token = sum(wl.heads)              # every normed tensor of a token (Q and K heads)
    times, rows_done = [], []
    with cf.ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
        def one(seconds):
            jobs = [(x[i * per:(i + 1) * per], dy[i * per:(i + 1) * per], w, wl.eps, seconds) for i in range(cores)]
            res = list(ex.map(_oracle_worker, jobs))
            return sum(r[0] for r in res), max(r[1] for r in res)
        for _ in range(args.warmup):
            one(0.05)
        for _ in range(args.steps):
            done, dt = one(per_step)
            times.append(dt)
            rows_done.append(done)
    tok_s = (sum(rows_done) / rows_per_token) / sum(times)
    sample = (f"{n_rows} logical rows of {wl.name} (hidden {H}); one spawned process per host core ({cores}), "
              f"each cycling its own slice of {per} rows for ~{per_step:.1f} s per step; a token is "
              f"{rows_per_token} such rows; FP64 C oracle (single-threaded code, unchanged)")
    ms = statistics.mean(times) * 1e3
    line = {"metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_desc(wl, lay_name, lay.n_physical), "hidden": H,
                       "heads": list(wl.heads), "tokens": wl.n_tokens, "layout": lay_name, "calls": len(lay.calls),
                       "l2": "not applicable: the oracle runs on the host, in logical order",
                       "launch": f"oracle calls on the host (FP64 C), one process per core ({cores})",
                       "parallelism": f"{cores} host processes"},
            "cpu_baseline": {"value": round(tok_s, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(tok_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

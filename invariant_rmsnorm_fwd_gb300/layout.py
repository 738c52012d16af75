"""Layout mapper: places a logical token multiset into physical calls.

A token is identified by (sample_id, position).  Its canonical logical id is
g = off[sample_id] + position, where off is the prefix sum of the sample
lengths in sample_id order, so the id does not depend on where or in which
call the token is placed ("[WS1 Closeout][Backward] ...", RL-Kernel #270,
Scope: compare on the same logical sample/token multiset; "WS1 C4 (#270)
closeout evidence": upstream gradients are a pure function of logical
identity, inactive tokens contribute 0).

A physical layout is a list of calls; each call is an int32 array tok_id over
its token slots (-1 = inactive padding slot).  The layout cells of "WS1 C4
(#270) closeout evidence", section "The matrix is falsifiable", are built
here: BN/full (one packed call), BN/chunked (the packed stream cut into
calls by row counts), B1 singleton (one call per sample), BN/padded_right and
BN/padded_left (every sample in a fixed-length slot), BN/permuted (samples
in a permuted order), plus the composites the workloads need (padding or
slots combined with chunking and permutation).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

LAYOUT_KINDS = ("full", "chunked", "singleton", "padded_right", "padded_left", "permuted")


@dataclass
class Layout:
    name: str
    calls: list                         # list of np.int32 arrays (tok_id per call)
    n_logical_tokens: int
    meta: dict = field(default_factory=dict)

    @property
    def rows_per_call(self):
        return [int(c.shape[0]) for c in self.calls]

    @property
    def n_physical(self) -> int:
        return int(sum(c.shape[0] for c in self.calls))

    def check_partition(self) -> None:
        """Every logical id appears exactly once over all calls."""
        ids = np.concatenate([c[c >= 0] for c in self.calls]) if self.calls else np.zeros(0, np.int32)
        if ids.size != self.n_logical_tokens or not np.array_equal(np.sort(ids), np.arange(self.n_logical_tokens)):
            raise ValueError(f"layout {self.name} is not a partition of the multiset")


def logical_offsets(lengths) -> np.ndarray:
    """off[s] = sum of lengths of samples with a smaller sample_id."""
    lengths = np.asarray(lengths, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)


def sample_ids(lengths, s: int) -> np.ndarray:
    off = logical_offsets(lengths)
    return (off[s] + np.arange(int(lengths[s]))).astype(np.int32)


def physical_stream(lengths, order=None, slot=None, pad_side: str = "right") -> np.ndarray:
    """Concatenate samples in `order`; with `slot` (int, or array per sample id)
    every sample sits in a slot of that many rows, padding on `pad_side`."""
    lengths = np.asarray(lengths, dtype=np.int64)
    order = np.arange(len(lengths)) if order is None else np.asarray(order)
    parts = []
    for s in order:
        ids = sample_ids(lengths, int(s))
        if slot is not None:
            sl = int(slot if np.isscalar(slot) else slot[s])
            pad = np.full(sl - ids.size, -1, dtype=np.int32)
            if pad.size < 0:
                raise ValueError("slot shorter than sample")
            ids = np.concatenate([ids, pad] if pad_side == "right" else [pad, ids])
        parts.append(ids)
    return np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)


def split_rows(stream: np.ndarray, chunk) -> list:
    """Cut a stream into consecutive calls: `chunk` is a row count or a list of counts."""
    if np.isscalar(chunk):
        chunk = int(chunk)
        return [stream[i:i + chunk] for i in range(0, stream.size, chunk)] or [stream[:0]]
    sizes = [int(c) for c in chunk]
    if sum(sizes) != stream.size:
        raise ValueError(f"chunk sizes sum to {sum(sizes)}, stream has {stream.size} rows")
    bounds = np.cumsum([0] + sizes)
    return [stream[bounds[i]:bounds[i + 1]] for i in range(len(sizes))]


def make_layout(kind: str, lengths, *, chunk=1024, perm=None, slot=None, per_sample_chunks=False,
                pad_side="right") -> Layout:
    """Build one layout of the multiset given by `lengths` (index = sample_id).

    kind: full | chunked | singleton | padded_right | padded_left | permuted |
          padded_right_chunked | permuted_slots_left_chunked | slots_left | permuted_chunked
    chunk: rows per call (int) or an explicit list of row counts.
    perm: sample order for permuted layouts (default: reversal).
    slot: slot length (int) or per-sample slot lengths; default the longest sample.
    per_sample_chunks: chunk each sample separately (chunks never cross samples).
    """
    lengths = np.asarray(lengths, dtype=np.int64)
    n = int(lengths.sum())
    S = len(lengths)
    if perm is None:
        perm = np.arange(S)[::-1].copy()
    if slot is None:
        slot = int(lengths.max()) if S else 0
    if kind == "full":
        calls = [physical_stream(lengths)]
    elif kind == "chunked":
        if per_sample_chunks:
            calls = []
            for s in range(S):
                calls += split_rows(sample_ids(lengths, s), chunk)
        else:
            calls = split_rows(physical_stream(lengths), chunk)
    elif kind == "singleton":
        calls = [sample_ids(lengths, s) for s in range(S)]
    elif kind in ("padded_right", "padded_left"):
        calls = [physical_stream(lengths, slot=slot, pad_side=kind.split("_")[1])]
    elif kind == "permuted":
        calls = [physical_stream(lengths, order=perm)]
    elif kind == "permuted_chunked":
        calls = split_rows(physical_stream(lengths, order=perm), chunk)
    elif kind == "padded_right_chunked":
        calls = split_rows(physical_stream(lengths, slot=slot, pad_side="right"), chunk)
    elif kind == "slots_left":
        calls = [physical_stream(lengths, slot=slot, pad_side="left")]
    elif kind == "permuted_slots_left_chunked":
        calls = split_rows(physical_stream(lengths, order=perm, slot=slot, pad_side="left"), chunk)
    else:
        raise KeyError(kind)
    lay = Layout(kind, [np.ascontiguousarray(c, dtype=np.int32) for c in calls], n)
    lay.check_partition()
    return lay


def workload_layouts(wl, kinds=None) -> dict:
    """The layouts of a workload (synth.Workload): the six cells, plus its headline layout."""
    import synth
    lengths = wl.lengths
    perm = synth.seeded_permutation(wl.seed, len(lengths))
    slot = wl.extra.get("slot")
    if wl.slot_factor:
        slot = (wl.slot_factor * lengths).astype(np.int64)
    per_sample = bool(wl.extra.get("per_sample_chunks", False))
    kinds = list(kinds) if kinds is not None else list(LAYOUT_KINDS) + (
        [wl.headline] if wl.headline not in LAYOUT_KINDS else [])
    out = {}
    for k in kinds:
        kw = dict(chunk=wl.chunk_rows, perm=perm, per_sample_chunks=per_sample)
        if k in ("padded_right", "padded_left", "padded_right_chunked") and slot is not None:
            kw["slot"] = slot
        if k in ("slots_left", "permuted_slots_left_chunked"):
            kw["slot"] = slot if slot is not None else None
        out[k] = make_layout(k, lengths, **kw)
    return out


def scatter_rows(logical: np.ndarray, tok_id: np.ndarray, fill) -> np.ndarray:
    """Physical copy of logical rows for one call: row t <- logical[tok_id[t]], padding <- fill."""
    out = np.empty((tok_id.size,) + logical.shape[1:], dtype=logical.dtype)
    out[...] = fill
    act = tok_id >= 0
    out[act] = logical[tok_id[act]]
    return out

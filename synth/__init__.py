"""Seeded synthetic inputs for the batch-invariant RMSNorm workloads.

This module is shared by the CUDA path's tests and bench and by the FP64
oracle's tests.  It holds only random-number generation, the workload
shapes (sample lengths, hidden sizes, heads) and the rounding of generated
values to bf16.  It computes nothing of RMSNorm itself.

Every value is a pure function of (seed, tensor tag, logical row, column):
a logical row is the canonical id of a (sample_id, position) token (times
the head count for per-head norms), so a token gets the same bits in every
physical layout.  The counter-based generator is SplitMix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014), and
normals come from the Box-Muller transform in float64.
"""
from __future__ import annotations

import math
import dataclasses
from dataclasses import dataclass, field

import numpy as np
import torch

# tensor tags: independent streams per tensor
TAG_X, TAG_W, TAG_DY, TAG_LEN, TAG_OUTLIER, TAG_PERM, TAG_WK = 1, 2, 3, 4, 5, 6, 7
TAG_RES, TAG_DRES = 8, 9          # residual-add chain: the residual input and its gradient
_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit constant as a signed int64 value."""
    v &= (1 << 64) - 1
    return v - (1 << 64) if v >= (1 << 63) else v


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 lanes (torch's >> is arithmetic)."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def splitmix64(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 finaliser of (z + golden gamma), on int64 lanes, wrapping."""
    z = z + _s64(_GOLDEN)
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def _key(seed: int, tag: int) -> int:
    z = torch.tensor([_s64(seed * 1000003 + tag)], dtype=torch.int64)
    return int(splitmix64(splitmix64(z))[0])


def uniform(seed: int, tag: int, rows: torch.Tensor, cols: torch.Tensor) -> torch.Tensor:
    """float64 uniforms in (0, 1) for the grid rows x cols (int64 tensors)."""
    base = splitmix64(rows.to(torch.int64).reshape(-1, 1) + _key(seed, tag))
    z = splitmix64(base + cols.to(torch.int64).reshape(1, -1).to(base.device))
    top53 = _lsr(z, 11).to(torch.float64)
    return (top53 + 0.5) * (1.0 / 9007199254740992.0)


def normal(seed: int, tag: int, rows: torch.Tensor, ncols: int) -> torch.Tensor:
    """float64 standard normals (Box-Muller, cosine branch) for rows x [0, ncols)."""
    cols = torch.arange(ncols, dtype=torch.int64, device=rows.device)
    u1 = uniform(seed, tag, rows, 2 * cols)
    u2 = uniform(seed, tag, rows, 2 * cols + 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def to_bf16(v: torch.Tensor) -> torch.Tensor:
    return v.to(torch.float32).to(torch.bfloat16)


def uniform_scalars(seed: int, tag: int, n: int) -> np.ndarray:
    rows = torch.arange(n, dtype=torch.int64)
    return uniform(seed, tag, rows, torch.zeros(1, dtype=torch.int64))[:, 0].numpy()


# ---------------------------------------------------------------- lengths

def lengths_uniform(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    u = uniform_scalars(seed, TAG_LEN, n)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64).clip(lo, hi)


def lengths_loguniform(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    u = uniform_scalars(seed, TAG_LEN, n)
    v = np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))
    return np.rint(v).astype(np.int64).clip(lo, hi)


def lengths_zipf_rescaled(seed: int, n: int, s: float, kmax: int, total: int) -> np.ndarray:
    """n draws of a Zipf(s) law truncated to [1, kmax] (inverse CDF), then
    rescaled with largest-remainder rounding so they sum to `total`, each >= 1."""
    k = np.arange(1, kmax + 1, dtype=np.float64)
    cdf = np.cumsum(k ** (-s))
    cdf /= cdf[-1]
    u = uniform_scalars(seed, TAG_LEN, n)
    raw = np.searchsorted(cdf, u, side="left").astype(np.int64) + 1
    raw = raw.clip(1, kmax).astype(np.float64)
    assert n <= total <= n * kmax

    def clipped(a):
        return np.clip(raw * a, 1.0, float(kmax))

    lo, hi = 0.0, float(kmax)          # scale factor alpha: sum(clipped(alpha)) is monotone
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if clipped(mid).sum() < total:
            lo = mid
        else:
            hi = mid
    ideal = clipped(hi)
    base = np.floor(ideal).astype(np.int64).clip(1, kmax)
    rem = total - int(base.sum())
    order = np.argsort(-(ideal - np.floor(ideal)), kind="stable")
    i = 0
    while rem != 0:                     # largest remainder first, respecting [1, kmax]
        j = order[i % n]
        if rem > 0 and base[j] < kmax:
            base[j] += 1
            rem -= 1
        elif rem < 0 and base[j] > 1:
            base[j] -= 1
            rem += 1
        i += 1
    assert int(base.sum()) == total and base.min() >= 1 and base.max() <= kmax
    return base


def seeded_permutation(seed: int, n: int) -> np.ndarray:
    """A non-identity permutation of range(n) (for n > 1), keyed by seed."""
    u = uniform_scalars(seed, TAG_PERM, n)
    p = np.argsort(u, kind="stable")
    if n > 1 and np.all(p == np.arange(n)):
        p = p[::-1].copy()
    return p


# ---------------------------------------------------------------- configs

@dataclass
class Workload:
    """One synthetic workload: sample lengths, hidden size, value recipe and layouts."""
    name: str
    hidden: int
    lengths: np.ndarray
    eps: float = 1e-6
    heads: tuple = (1,)                 # rows per token of each normed tensor (qk: (32, 8))
    x_std: float = 1.0
    dy_std: float = 1e-2
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    chunk_rows: object = 1024           # int, or an explicit list of row counts
    slot_factor: int = 0                # >0: each sample occupies slot_factor*len rows
    headline: str = "full"
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def n_tokens(self) -> int:
        return int(np.sum(self.lengths))


def truncated(wl: Workload, max_tokens: int) -> Workload:
    """The same workload cut to its first max_tokens logical tokens (samples in
    sample_id order, the last one shortened); values are unchanged because they
    are keyed by logical id.  Used for profiling runs of a smaller size."""
    out, left = [], int(max_tokens)
    for n in wl.lengths:
        if left <= 0:
            break
        out.append(min(int(n), left))
        left -= out[-1]
    return dataclasses.replace(wl, name=f"{wl.name}[:{int(max_tokens)}]", lengths=np.asarray(out, dtype=np.int64))


def config(name: str, seed: int = 0) -> Workload:
    """The five workloads of the benchmark plus the pages' own worked layout.

    c0  hidden=8, 8 samples [10,7,9,5,8,6,10,4] (59 tokens), dy ~ N(0,1).
    c0p hidden=8, 4 samples [11,16,13,19] (59 tokens): the pages' worked layout.
    c1  hidden=4096, 8 samples with lengths uniform in [512,4096], chunk 1024.
    c2  hidden=8192, 32 samples log-uniform in [64,8192], x ~ N(0,2) with 1%
        outlier rows x30, right-padded to the longest sample, chunk 2048.
    c3  per-head norm, head_dim=128, Q 32 heads and K 8 heads, 16 samples
        uniform in [256,4096], chunk 1024 tokens.
    c4  hidden=5120, 256 samples Zipf(1.2) in [1,16384] rescaled to 2^18
        tokens, slots of 4x the length (25% active), left-padded, chunk 4096.
    """
    if name == "c0":
        return Workload("c0", 8, np.array([10, 7, 9, 5, 8, 6, 10, 4]), dy_std=1.0,
                        chunk_rows=[7, 4, 7, 7, 2, 7, 6, 7, 7, 5], seed=seed)
    if name == "c0p":
        return Workload("c0p", 8, np.array([11, 16, 13, 19]), dy_std=1.0,
                        chunk_rows=7, seed=seed, extra={"per_sample_chunks": True, "slot": 20})
    if name == "c1":
        return Workload("c1", 4096, lengths_uniform(seed + 1, 8, 512, 4096),
                        chunk_rows=1024, seed=seed)
    if name == "c2":
        return Workload("c2", 8192, lengths_loguniform(seed + 2, 32, 64, 8192),
                        x_std=2.0, outlier_frac=0.01, outlier_scale=30.0,
                        chunk_rows=2048, headline="padded_right_chunked", seed=seed)
    if name == "c3":
        return Workload("c3", 128, lengths_uniform(seed + 3, 16, 256, 4096),
                        heads=(32, 8), chunk_rows=1024, seed=seed)
    if name == "c4":
        return Workload("c4", 5120, lengths_zipf_rescaled(seed + 4, 256, 1.2, 16384, 1 << 18),
                        chunk_rows=4096, slot_factor=4,
                        headline="permuted_slots_left_chunked", seed=seed)
    raise KeyError(name)


# ---------------------------------------------------------------- values

def weight(wl: Workload, head_set: int = 0, device="cpu") -> torch.Tensor:
    """w = 1 + 0.1*N(0,1), bf16 [hidden]; head_set selects Q (0) or K (1) weights."""
    tag = TAG_W if head_set == 0 else TAG_WK
    n = normal(wl.seed, tag, torch.zeros(1, dtype=torch.int64, device=device), wl.hidden)[0]
    return to_bf16(1.0 + 0.1 * n)


def logical_rows(wl: Workload, rows: torch.Tensor, tag: int, std: float,
                 head_set: int = 0) -> torch.Tensor:
    """bf16 values of the given logical rows, N(0, std) (std is a standard deviation)."""
    t = tag + 16 * head_set
    v = normal(wl.seed, t, rows, wl.hidden) * std
    if tag == TAG_X and wl.outlier_frac > 0:
        u = uniform(wl.seed, TAG_OUTLIER + 16 * head_set, rows,
                    torch.zeros(1, dtype=torch.int64, device=rows.device))[:, 0]
        v = torch.where((u < wl.outlier_frac).reshape(-1, 1), v * wl.outlier_scale, v)
    return to_bf16(v)


def logical_tensor(wl: Workload, tag: int, n_rows: int, std: float, head_set: int = 0,
                   device="cpu", chunk: int = 4096) -> torch.Tensor:
    """All n_rows logical rows in canonical order, bf16 [n_rows, hidden], generated in
    row chunks on `device` (values do not depend on the chunking)."""
    out = torch.empty((n_rows, wl.hidden), dtype=torch.bfloat16, device=device)
    for r0 in range(0, n_rows, chunk):
        r1 = min(n_rows, r0 + chunk)
        rows = torch.arange(r0, r1, dtype=torch.int64, device=device)
        out[r0:r1] = logical_rows(wl, rows, tag, std, head_set)
    return out


def poison_bf16(shape, device="cpu") -> torch.Tensor:
    """bf16 NaN fill for inactive (padding) rows: any leak shows up in the outputs."""
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device=device)

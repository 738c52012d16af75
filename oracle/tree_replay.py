"""FP32 replay of the weight-gradient reduction order (TEST INFRASTRUCTURE ONLY).

The weight gradient is a sum of per-logical-row FP32 contributions
c_g = dy_g * xhat_g ("WS1 C4 (#270) closeout evidence", opening note and
"Historical finding - RMSNorm dweight is not chunk/batch decomposable":
the fix reduces logical-row FP32 contributions instead of a fold whose
shape follows the row count of a call).  The pages fix no reduction tree;
the benchmark statement fixes this one, replayed here step by step:

1. Logical rows are grouped in blocks of 64 consecutive logical ids; block b
   holds ids [64b, 64b+64).  Ids at or beyond N are leaves equal to +0.0.
2. Each block is reduced by a complete pairwise tree over its 64 leaves in
   logical order: level 1 adds (0,1), (2,3), ...; level 2 adds adjacent
   level-1 results; six levels in all.
3. The nb = ceil(N/64) block partials are reduced by a pairwise tree: at each
   level element 2i is added to element 2i+1, and an odd last element is
   carried up unchanged; until one value remains.

Every addition is one IEEE binary32 round-to-nearest-even addition (numpy
float32).  Leaves are given, so this replays only the order of the sum.
"""
from __future__ import annotations

import numpy as np

BLOCK = 64


def pairwise_levels(v: np.ndarray) -> np.ndarray:
    """Pairwise tree along axis 0 with odd carry, level by level (float32)."""
    v = np.asarray(v, dtype=np.float32)
    while v.shape[0] > 1:
        m = v.shape[0]
        pairs = v[0:m - (m % 2):2] + v[1:m - (m % 2):2]   # element-wise float32 adds
        if m % 2:
            pairs = np.concatenate([pairs, v[m - 1:m]], axis=0)
        v = pairs.astype(np.float32)
    return v[0]


def block_partials(leaves: np.ndarray) -> np.ndarray:
    """[nb, H] block partials of float32 leaves [N, H] (steps 1-2)."""
    leaves = np.asarray(leaves, dtype=np.float32)
    n, H = leaves.shape
    nb = (n + BLOCK - 1) // BLOCK
    padded = np.zeros((nb * BLOCK, H), dtype=np.float32)      # +0.0 beyond N
    padded[:n] = leaves
    out = np.empty((nb, H), dtype=np.float32)
    for b in range(nb):
        blk = padded[b * BLOCK:(b + 1) * BLOCK]
        assert blk.shape[0] == BLOCK                         # always complete: 6 levels
        out[b] = pairwise_levels(blk)
    return out


def dweight(leaves: np.ndarray) -> np.ndarray:
    """float32 [H] weight gradient in the fixed order (steps 1-3)."""
    leaves = np.asarray(leaves, dtype=np.float32)
    if leaves.shape[0] == 0:
        return np.zeros(leaves.shape[1], dtype=np.float32)
    return pairwise_levels(block_partials(leaves))

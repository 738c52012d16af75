"""Data-parallel weight gradient over several ranks, bitwise equal to one device.

The weight gradient of one logical multiset is a fixed tree: 64-row logical
blocks, then a pairwise tree with odd carry over the block partials (the
statement of batch-invariant RMSNorm that the pages' fix follows: "WS1 C4
(#270) closeout evidence", "Historical finding - RMSNorm dweight is not
chunk/batch decomposable", where the cure is to reduce logical-row FP32
contributions in an order that no call shape decides).  In that tree, a
range of 2^k blocks starting at a multiple of 2^k is one node, and the last
such range, cut at the block count, is the node that carries the odd tail.
So the blocks are split into consecutive ranges of one size 2^k, each rank
owns a run of consecutive ranges (and the logical rows in them), reduces each
of its ranges to its node on its own device, and the ranks exchange only the
nodes: one all-gather of at most a few rows of FP32 [H] per rank.  Every rank
then forms the same top of the tree with dweight_combine.  No all-reduce is
used, since its summation order belongs to the collective library.

Rows and x/dy of a rank's shard are numbered locally from the rank's first
row; the shard boundaries are token boundaries, so a rank runs any physical
layout of its tokens (packed, chunked, padded, permuted) with local ids.
"""
from __future__ import annotations

from dataclasses import dataclass

BLOCK_ROWS = 64
MAX_ROOTS = 2047            # dweight_combine takes fewer than 2048 roots


@dataclass(frozen=True)
class ShardPlan:
    n_logical_tokens: int
    rows_per_token: int
    world_size: int
    block_count: int         # blocks per range: a power of two
    n_ranges: int
    rank_ranges: tuple       # per rank: (first range, end range), consecutive

    @property
    def n_rows(self) -> int:
        return self.n_logical_tokens * self.rows_per_token

    @property
    def n_blocks(self) -> int:
        return (self.n_rows + BLOCK_ROWS - 1) // BLOCK_ROWS

    @property
    def max_ranges_per_rank(self) -> int:
        return max((b - a for a, b in self.rank_ranges), default=0)

    def rows(self, rank: int):
        """Logical rows [lo, hi) of this rank."""
        a, b = self.rank_ranges[rank]
        span = self.block_count * BLOCK_ROWS
        return min(a * span, self.n_rows), min(b * span, self.n_rows)

    def tokens(self, rank: int):
        """Logical tokens [lo, hi) of this rank (row bounds are token bounds)."""
        lo, hi = self.rows(rank)
        return lo // self.rows_per_token, hi // self.rows_per_token

    def local_ranges(self, rank: int):
        """(block_lo, block_count) of each of this rank's ranges in its local workspace."""
        a, b = self.rank_ranges[rank]
        return [((j - a) * self.block_count, self.block_count) for j in range(a, b)]


def plan_shards(n_logical_tokens: int, rows_per_token: int, world_size: int,
                ranges_per_rank: int = 4) -> ShardPlan:
    """Split the blocks of N = n_logical_tokens * rows_per_token logical rows into
    ranges of 2^k blocks (k the smallest with at most ranges_per_rank ranges per
    rank on average and fewer than 2048 ranges in all, and with token bounds at
    range bounds), then give each rank a balanced run of consecutive ranges."""
    N = int(n_logical_tokens) * int(rows_per_token)
    R = int(rows_per_token)
    if world_size < 1 or R < 1 or n_logical_tokens < 0 or ranges_per_rank < 1:
        raise ValueError("bad shard request")
    nb = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    if world_size > 1 and (R & (R - 1)) != 0:
        raise ValueError(f"rows_per_token={R}: rank bounds must be token bounds; only powers of two are sharded")
    bc = 1
    while True:
        nr = (nb + bc - 1) // bc
        if (nr <= max(1, world_size * ranges_per_rank) and nr <= MAX_ROOTS
                and (world_size == 1 or (bc * BLOCK_ROWS) % R == 0)):
            break
        bc *= 2
    ranges = tuple((r * nr // world_size, (r + 1) * nr // world_size) for r in range(world_size))
    return ShardPlan(int(n_logical_tokens), R, int(world_size), bc, nr, ranges)


def local_roots(workspace, plan: ShardPlan, rank: int, stream=None):
    """FP32 [ranges of this rank, H] nodes of the rank's ranges, from its local workspace
    (begun for plan.rows(rank) rows and filled with the backward of its tokens)."""
    import torch
    lr = plan.local_ranges(rank)
    out = torch.empty(len(lr), workspace.hidden, dtype=torch.float32, device=workspace.buf.device)
    for i, (lo, cnt) in enumerate(lr):
        workspace.finalize_range(lo, cnt, root=out[i], stream=stream)
    return out


def assemble_roots(per_rank, plan: ShardPlan):
    """Roots of all ranges in block order from the ranks' (possibly padded) root rows."""
    import torch
    parts = []
    for r, (a, b) in enumerate(plan.rank_ranges):
        parts.append(per_rank[r][:b - a])
    return torch.cat(parts, dim=0).contiguous()


def gather_roots(local, plan: ShardPlan, group=None):
    """All-gather of every rank's roots; each rank gets all roots in block order.

    The one exchange of the sharded backward.  Rows are padded to the largest
    per-rank count so that one fixed-size all-gather suffices.  With the gloo
    backend the exchange goes through host memory."""
    import torch
    import torch.distributed as dist
    H = local.shape[1]
    m = max(plan.max_ranges_per_rank, 1)
    via_host = dist.get_backend(group) == "gloo"
    dev = local.device
    buf = torch.zeros(m, H, dtype=torch.float32, device="cpu" if via_host else dev)
    buf[:local.shape[0]] = local.to(buf.device)
    bufs = [torch.empty_like(buf) for _ in range(plan.world_size)]
    dist.all_gather(bufs, buf, group=group)
    return assemble_roots(bufs, plan).to(dev)


def gather_status(status: int, group=None) -> int:
    """Bitwise OR of the ranks' workspace status words."""
    import torch
    import torch.distributed as dist
    via_host = dist.get_backend(group) == "gloo"
    t = torch.tensor([int(status)], dtype=torch.int64,
                     device="cpu" if via_host else f"cuda:{torch.cuda.current_device()}")
    out = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(out, t, group=group)
    s = 0
    for o in out:
        s |= int(o.item())
    return s


def sharded_dweight(workspace, plan: ShardPlan, rank: int, group=None, stream=None, grad_scale: float = 1.0):
    """dweight of the whole multiset on every rank, bitwise equal to one device's
    dweight_finalize_scaled over all rows: local nodes, all-gather, combine."""
    import torch
    from . import dweight_combine
    if plan.n_ranges == 0:
        return torch.zeros(workspace.hidden, dtype=torch.float32, device=workspace.buf.device)
    roots = gather_roots(local_roots(workspace, plan, rank, stream), plan, group)
    return dweight_combine(roots.to(workspace.buf.device), stream=stream, grad_scale=grad_scale)

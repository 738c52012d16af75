"""Sharded weight gradient across ranks: plan, node property, all-gather (CPU).

The node property is checked with the oracle's FP32 tree replay, whose
order is the benchmark statement's: 64-row blocks, then a pairwise tree with
odd carry.  Leaves are drawn with exponents spread over many binades, so any
other association order changes FP32 bits and a wrong split fails.  The
exchange itself runs as gloo ranks (world sizes 2 and 3) on the host.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from invariant_rmsnorm_fwd_gb300 import sharded as S
from oracle import tree_replay


def _leaves(n, H, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(n, H)) * np.exp2(rng.integers(-20, 20, size=(n, H)))).astype(np.float32)


def _rank_roots(leaves, plan, rank):
    """Roots of the rank's ranges computed from its own rows only (local numbering)."""
    lo, hi = plan.rows(rank)
    if hi <= lo:
        return np.zeros((0, leaves.shape[1]), np.float32)
    parts = tree_replay.block_partials(leaves[lo:hi])
    return np.stack([tree_replay.pairwise_levels(parts[b:b + c]) for b, c in plan.local_ranges(rank)])


@pytest.mark.parametrize("n_tokens,rpt", [(0, 1), (1, 1), (59, 1), (64, 1), (65, 1), (1000, 1), (18000, 1),
                                          (4097, 32), (300, 8), (262144, 1)])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_plan_covers_blocks_with_aligned_ranges(n_tokens, rpt, world):
    p = S.plan_shards(n_tokens, rpt, world)
    bc = p.block_count
    assert bc & (bc - 1) == 0 and p.n_ranges <= S.MAX_ROOTS
    assert p.n_ranges == (p.n_blocks + bc - 1) // bc
    assert p.rank_ranges[0][0] == 0 and p.rank_ranges[-1][1] == p.n_ranges
    for (a0, b0), (a1, _) in zip(p.rank_ranges, p.rank_ranges[1:]):
        assert b0 == a1 and a0 <= b0
    counts = [b - a for a, b in p.rank_ranges]
    assert max(counts) - min(counts) <= 1                              # balanced
    rows = [p.rows(r) for r in range(world)]
    assert rows[0][0] == 0 and rows[-1][1] == n_tokens * rpt
    for (lo, hi), (lo2, _) in zip(rows, rows[1:]):
        assert hi == lo2
    for lo, hi in rows:
        assert lo % rpt == 0 and hi % rpt == 0                       # token bounds
    for r in range(world):
        for b, c in p.local_ranges(r):
            assert c == bc and b % c == 0


def test_plan_rejects_what_cannot_be_sharded():
    with pytest.raises(ValueError):
        S.plan_shards(100, 40, 2)                                    # 40 rows per token never meets 64 * 2^k
    assert S.plan_shards(100, 40, 1).n_ranges >= 1                   # one rank needs no bound
    with pytest.raises(ValueError):
        S.plan_shards(10, 1, 0)


@pytest.mark.parametrize("n", [1, 63, 64, 65, 129, 1000, 4160, 9000])
@pytest.mark.parametrize("world", [1, 2, 3, 5, 8])
def test_aligned_ranges_are_nodes_of_the_tree(n, world):
    H = 4
    leaves = _leaves(n, H, seed=n * 10 + world)
    want = tree_replay.dweight(leaves)
    p = S.plan_shards(n, 1, world, ranges_per_rank=3)
    roots = np.concatenate([_rank_roots(leaves, p, r) for r in range(world)])
    assert roots.shape[0] == p.n_ranges
    got = tree_replay.pairwise_levels(roots)
    assert got.tobytes() == want.tobytes()


def test_unaligned_split_is_not_a_node():
    """Control: cutting the blocks at a non-aligned point changes the bits."""
    leaves = _leaves(64 * 7, 64, seed=3)
    parts = tree_replay.block_partials(leaves)
    want = tree_replay.dweight(leaves)
    bad = tree_replay.pairwise_levels(np.stack([tree_replay.pairwise_levels(parts[:3]),
                                                tree_replay.pairwise_levels(parts[3:])]))
    assert bad.tobytes() != want.tobytes()


def test_assemble_roots_drops_padding_rows():
    p = S.ShardPlan(640, 1, 3, 1, 10, ((0, 3), (3, 6), (6, 10)))
    per = [torch.full((4, 2), float(r)) for r in range(3)]
    for r in range(3):
        per[r][:, 1] = torch.arange(4, dtype=torch.float32)
    out = S.assemble_roots(per, p)
    assert out[:, 0].tolist() == [0, 0, 0, 1, 1, 1, 2, 2, 2, 2]
    assert out[:, 1].tolist() == [0, 1, 2, 0, 1, 2, 0, 1, 2, 3]


def _worker(rank, world, port, n, H, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        leaves = _leaves(n, H, seed=11)
        p = S.plan_shards(n, 1, world, ranges_per_rank=2)
        local = torch.as_tensor(_rank_roots(leaves, p, rank))
        roots = S.gather_roots(local, p)
        dw = tree_replay.pairwise_levels(roots.numpy())
        status = S.gather_status(4 if rank == world - 1 else 0)
        np.save(os.path.join(out_dir, f"dw{rank}.npy"), dw)
        np.save(os.path.join(out_dir, f"st{rank}.npy"), np.array([status]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_reach_the_single_device_tree(world, tmp_path):
    n, H = 1000, 16
    port = 29500 + (os.getpid() % 2000) + world
    mp.start_processes(_worker, args=(world, port, n, H, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    want = tree_replay.dweight(_leaves(n, H, seed=11))
    for r in range(world):
        assert np.load(tmp_path / f"dw{r}.npy").tobytes() == want.tobytes()
        assert int(np.load(tmp_path / f"st{r}.npy")[0]) == 4

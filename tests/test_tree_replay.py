"""Pins of the FP32 reduction-order replay against hand-worked binary32 sums
(tests/golden/tree_examples.json) and against exact sums."""
import json
import os

import numpy as np
import pytest

from oracle import tree_replay

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _val(v):
    return np.float32(float(v)) if not isinstance(v, str) else np.float32(float(v.replace("+", "")))


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "tree_examples.json")))["cases"],
                         ids=lambda c: c["name"])
def test_hand_worked_trees(case):
    n = case["n"]
    leaves = np.zeros((n, 1), dtype=np.float32)
    if "leaves_all" in case:
        leaves[:] = _val(case["leaves_all"])
    for k, v in case.get("leaves", {}).items():
        leaves[int(k), 0] = _val(v)
    got = tree_replay.dweight(leaves)[0]
    want = _val(case["expected"])
    assert got.tobytes() == want.tobytes(), (got, want)


def test_exact_sums_match_integer_arithmetic():
    rng = np.random.default_rng(5)
    for n in (1, 63, 64, 65, 130, 1000):
        ints = rng.integers(-1000, 1000, size=(n, 3))
        got = tree_replay.dweight(ints.astype(np.float32))
        assert np.array_equal(got, ints.sum(axis=0).astype(np.float32))


def test_block_partials_are_per_block():
    leaves = np.arange(200, dtype=np.float32).reshape(200, 1)
    p = tree_replay.block_partials(leaves)
    assert p.shape == (4, 1)
    assert p[0, 0] == np.arange(64).sum() and p[3, 0] == np.arange(192, 200).sum()


def test_empty_multiset_gives_zero():
    assert np.array_equal(tree_replay.dweight(np.zeros((0, 5), np.float32)), np.zeros(5, np.float32))

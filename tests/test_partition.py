"""Load-balanced partition over training workers (AREAL-DTA, section 4).

Oracle pins (the oracle checked against something other than itself) and the
library's partitioner checked against the oracle.  CPU only.
"""
import json
import os

import numpy as np
import pytest

import workloads as W
from oracle import partition as OP
from oracle import trie as OT

import prefix_tree_attention_gb300 as ptg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def _random_sets(n_sets, max_seqs, max_len, alphabet, seed):
    rng = W.SplitMix64(seed)
    for _ in range(n_sets):
        yield W.random_sequences(rng, rng.randint(1, max_seqs), max_len, alphabet)


# ------------------------------------------------------------ oracle pins
def test_tree_tokens_worked_example():
    g = json.load(open(GOLDEN))
    assert OP.tree_tokens(g["sequences"]) == g["n_tokens"] == 8


def test_tree_tokens_equals_oracle_trie_token_count():
    for seqs in _random_sets(200, 6, 6, 3, seed=11):
        (tr,) = OT.pack_sequences(seqs, 1024)
        assert OP.tree_tokens(seqs) == int((tr.token_node >= 0).sum())


def test_dfs_order_is_lexicographic_preorder():
    g = json.load(open(GOLDEN))
    # A B C D, A B E F, A G H: already in DFS order of the figure's trie
    assert OP.dfs_order(g["sequences"]) == [0, 1, 2]
    assert OP.dfs_order([[2], [1, 5], [1]]) == [2, 1, 0]


def test_optimal_contiguous_equals_exhaustive_enumeration():
    for seqs in _random_sets(120, 7, 4, 3, seed=12):
        order = OP.dfs_order(seqs)
        for k in (1, 2, 3, 4):
            brute = min(max(OP.tree_tokens([seqs[order[t]] for t in range(a, b)])
                            for a, b in split)
                        for split in OP.all_contiguous_splits(len(seqs), k))
            assert OP.optimal_contiguous(seqs, k) == brute


def test_worked_example_two_workers():
    g = json.load(open(GOLDEN))
    # {ABCD} | {ABEF, AGH} costs 4 and 6; {ABCD, ABEF} | {AGH} costs 6 and 3
    assert OP.optimal_contiguous(g["sequences"], 2) == 6
    assert OP.optimal_contiguous(g["sequences"], 3) == 4


# ------------------------------------------------------ library vs oracle
def _oracle_trie_tokens(group):
    """Token count of a group's tree from the oracle's trie packer (for
    inputs too long for the distinct-prefix count)."""
    if not group:
        return 0
    cap = -(-sum(len(s) for s in group) // 128) * 128
    (tr,) = OT.pack_sequences(group, cap)
    return int((tr.token_node >= 0).sum())


def _check_library(seqs, k, cost_fn=OP.tree_tokens):
    groups, cost, mx = ptg.partition_sequences(seqs, k)
    order = OP.dfs_order(seqs)
    along = [int(groups[i]) for i in order]
    assert along == sorted(along), "groups are not contiguous in DFS order"
    assert 0 <= min(along) and max(along) < k
    for gi in range(k):
        members = [seqs[i] for i in range(len(seqs)) if groups[i] == gi]
        assert int(cost[gi]) == cost_fn(members)
    assert mx == int(cost.max())
    return groups, cost, mx


def test_library_partition_is_optimal_for_the_dfs_order():
    for seqs in _random_sets(150, 9, 5, 3, seed=13):
        for k in (1, 2, 3, 4):
            _g, _c, mx = _check_library(seqs, k)
            assert mx == OP.optimal_contiguous(seqs, k)


def test_library_partition_worked_example():
    g = json.load(open(GOLDEN))
    groups, cost, mx = _check_library(g["sequences"], 2)
    assert mx == 6 and sorted(cost.tolist()) == [3, 6]


@pytest.mark.parametrize("key", ["agent", "tiny"])
def test_partition_of_a_workload(key):
    seqs = W.sequences(key)
    if key == "agent":
        seqs = seqs[:64]          # 8 tasks x 8 rollouts keeps the oracle packer quick
    whole = _oracle_trie_tokens(seqs)
    longest = max(len(s) for s in seqs)
    for k in (1, 2, 4, 8):
        groups, cost, mx = _check_library(seqs, k, _oracle_trie_tokens)
        # the page's bound on prefix sharing lost by cutting the DFS order
        assert int(cost.sum()) <= whole + (k - 1) * longest
        assert mx >= -(-whole // k)
        # each group packed alone by the library's packer is one trie of that size
        cap = -(-mx // 128) * 128
        for gi in range(k):
            members = [s for s, g in zip(seqs, groups) if g == gi]
            if not members:
                assert int(cost[gi]) == 0
                continue
            (tr,) = ptg.pack_sequences(members, cap)
            assert tr.n_tokens == int(cost[gi])


def test_partition_errors():
    with pytest.raises(ptg.TreeError):
        ptg.partition_sequences([[1, 2]], 0)
    with pytest.raises(ptg.TreeError):
        ptg.partition_sequences([[1, 2], []], 2)
    with pytest.raises(ptg.TreeError):
        ptg.partition_sequences([], 2)


def test_more_workers_than_sequences_leaves_empty_groups():
    groups, cost, mx = ptg.partition_sequences([[1, 2, 3], [4, 5]], 4)
    assert sorted(groups.tolist()) == [0, 1]
    assert cost.tolist()[2:] == [0, 0] and mx == 3

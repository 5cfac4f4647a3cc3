"""Oracle load-balanced partition — TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows AREAL-DTA, section 4 "负载均衡并行化" (load-balanced parallelisation):

* problem formalisation: N sequences are split into K disjoint groups, one
  per training worker; worker j builds one prefix tree T_j from its group,
  and the cost C(T_j) is the tree's token count (the sum of its nodes' token
  lengths).  The objective is min over splits of max_j C(T_j);
* the partition algorithm restricts the split to K contiguous segments of
  the sequences in DFS order of the single combined prefix tree, which the
  page obtains by lexicographic sorting.

What this module computes, each as the plain definition:

* ``tree_tokens(group)`` — the token count of the prefix tree of a group,
  counted directly as the number of distinct non-empty prefixes (every
  prefix is one token of the tree);
* ``dfs_order(seqs)`` — indices in lexicographic order of the token lists,
  ties by input index (Python's sort is stable);
* ``optimal_contiguous(seqs, K)`` — the exact minimum of max_j C(T_j) over
  every split of the DFS order into at most K contiguous segments, by
  dynamic programming over segment ends (costs recomputed from scratch per
  candidate segment; cubic time, small inputs only);
* ``all_contiguous_splits(n, K)`` — every such split, for exhaustive checks.

The page's own solution method (binary search on the bound with a greedy
scan) is what the library implements; tests check it against
``optimal_contiguous``.  Reading where the page is silent: fewer than K
non-empty segments are allowed ("at most K segments"); the remaining
workers get an empty group.

Parity: ``tree_tokens`` is pinned by the worked example of the tree-training
guide's packing figure (8 tokens) and by the oracle trie packer's token
count; ``optimal_contiguous`` by exhaustive enumeration of every split on
small inputs (tests/test_partition.py).
"""
from __future__ import annotations

import itertools


def tree_tokens(group) -> int:
    """Token count of the prefix tree built from the sequences of ``group``."""
    prefixes = set()
    for s in group:
        for n in range(1, len(s) + 1):
            prefixes.add(tuple(s[:n]))
    return len(prefixes)


def dfs_order(seqs) -> list:
    """Sequence indices in DFS order of their combined prefix tree."""
    return sorted(range(len(seqs)), key=lambda i: list(seqs[i]))


def optimal_contiguous(seqs, n_groups: int) -> int:
    """min over splits of the DFS order into <= n_groups contiguous
    segments of the largest segment tree cost."""
    order = dfs_order(seqs)
    n = len(order)
    inf = float("inf")
    # best[k][j]: smallest max cost splitting the first j sequences into k segments
    best = [[inf] * (n + 1) for _ in range(n_groups + 1)]
    best[0][0] = 0
    for k in range(1, n_groups + 1):
        for j in range(1, n + 1):
            for i in range(k - 1, j):
                if best[k - 1][i] == inf:
                    continue
                c = tree_tokens([seqs[order[t]] for t in range(i, j)])
                best[k][j] = min(best[k][j], max(best[k - 1][i], c))
    return int(min(best[k][n] for k in range(1, n_groups + 1)))


def all_contiguous_splits(n: int, n_groups: int):
    """Every split of range(n) into 1..n_groups contiguous non-empty
    segments, as lists of (start, end) pairs."""
    for k in range(1, min(n, n_groups) + 1):
        for cuts in itertools.combinations(range(1, n), k - 1):
            bounds = (0,) + cuts + (n,)
            yield [(bounds[t], bounds[t + 1]) for t in range(k)]

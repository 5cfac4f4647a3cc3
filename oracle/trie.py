"""Oracle trie packing — TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows the AReaL Tree Training guide, section "树构建流程" (tree
construction), in its order:

1. sequences arrive as plain token lists (step 1, "extract sequences");
2. first-fit-decreasing greedy packing: longest sequence first, each goes into
   the first trie whose occupied node count plus the nodes it would add stays
   within ``max_tokens_per_mb``, else a new trie is opened (step 2);
3. compression: a node with exactly one child whose passing-sequence set is
   identical to its own absorbs that child (step 3);
4. layout: nodes are flattened in preorder under a virtual root, each node's
   tokens contiguous (section "核心数据结构：TrieNode": ``start_idx``/
   ``end_idx`` inclusive, ``nodes`` in preorder, root holds no token), and the
   packed length is padded to a multiple of the 128-token block
   (section "FlexAttention + BlockMask").

Validation follows section "参数背后的源码校验逻辑": ``max_tokens_per_mb``
must be positive and a multiple of the block, and no sequence may be longer
than ``max_tokens_per_mb``.

Readings where the page is silent:
* children keep insertion order (the page keys children in a ``dict``);
* FFD sorts by length descending, ties by original index (stable sort);
* capacity counts uncompressed nodes, i.e. tokens;
* an empty sequence is rejected.

Parity: pinned by the worked example of the packing figure, by brute force
over every small sequence set (distinct-prefix count, span round trip,
positions along each sequence) and by the unpack invariant of the attention
oracle (tests/test_oracle_*.py).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


class Node:
    """One trie node: a run of tokens plus the ids of sequences passing it."""

    __slots__ = ("tokens", "seq_ids", "children", "parent")

    def __init__(self, parent):
        self.tokens: list[int] = []
        self.seq_ids: list[int] = []
        self.children: dict[int, Node] = {}   # first token of child -> child
        self.parent = parent


class Trie:
    """An uncompressed trie (one token per node) with a virtual root."""

    def __init__(self):
        self.root = Node(None)
        self.occupied = 0          # number of non-root nodes (= tokens)
        self.seq_ids: list[int] = []

    def additional_nodes(self, seq) -> int:
        """Nodes that inserting ``seq`` would add (its unmatched suffix)."""
        node = self.root
        matched = 0
        for tok in seq:
            child = node.children.get(tok)
            if child is None:
                break
            node = child
            matched += 1
        return len(seq) - matched

    def insert(self, seq, sid: int) -> None:
        node = self.root
        for tok in seq:
            child = node.children.get(tok)
            if child is None:
                child = Node(node)
                child.tokens = [tok]
                node.children[tok] = child
                self.occupied += 1
            child.seq_ids.append(sid)
            node = child
        self.seq_ids.append(sid)


def greedy_ffd(seqs, max_tokens_per_mb: int) -> list[Trie]:
    """Step 2: first-fit-decreasing insertion of sequences into tries."""
    order = sorted(range(len(seqs)), key=lambda i: (-len(seqs[i]), i))
    tries: list[Trie] = []
    for sid in order:
        seq = seqs[sid]
        placed = False
        for t in tries:
            if t.occupied + t.additional_nodes(seq) <= max_tokens_per_mb:
                t.insert(seq, sid)
                placed = True
                break
        if not placed:
            t = Trie()
            t.insert(seq, sid)
            tries.append(t)
    return tries


def compress(trie: Trie) -> None:
    """Step 3: merge single-child chains whose passing sequences are equal."""
    stack = list(trie.root.children.values())
    while stack:
        node = stack.pop()
        while len(node.children) == 1:
            (child,) = node.children.values()
            if sorted(child.seq_ids) != sorted(node.seq_ids):
                break
            node.tokens.extend(child.tokens)
            node.children = child.children
            for grandchild in node.children.values():
                grandchild.parent = node
        stack.extend(node.children.values())


@dataclass
class PackedTrie:
    """Flat preorder layout of one trie (all arrays int32, pads = -1)."""

    seq_ids: list[int]               # sequences in this trie, insertion order
    n_tokens: int                    # real (unpadded) tokens
    T_pad: int                       # padded length
    token_node: np.ndarray           # [T_pad] node of each token, -1 = pad
    token_ids: np.ndarray            # [T_pad] token id, -1 = pad
    node_entry: np.ndarray           # [N] preorder rank of the node
    node_exit: np.ndarray            # [N] largest preorder rank in its subtree
    node_parent: np.ndarray          # [N] parent node, -1 = child of root
    node_start: np.ndarray           # [N] first token index (inclusive)
    node_end: np.ndarray             # [N] last token index (inclusive)
    seq_index: dict = field(default_factory=dict)  # sid -> packed indices

    @property
    def n_nodes(self) -> int:
        return int(self.node_entry.shape[0])


def layout(trie: Trie, block: int = 128, pad_to: int | None = None) -> PackedTrie:
    """Step 4: preorder flattening under the virtual root, then padding."""
    preorder: list[Node] = []
    stack = list(reversed(list(trie.root.children.values())))
    while stack:
        node = stack.pop()
        preorder.append(node)
        stack.extend(reversed(list(node.children.values())))
    rank = {id(n): r for r, n in enumerate(preorder)}
    N = len(preorder)
    n_tokens = sum(len(n.tokens) for n in preorder)
    if pad_to is None:
        T_pad = -(-n_tokens // block) * block
    else:
        if pad_to % block or pad_to < n_tokens:
            raise ValueError("pad_to must be a block multiple >= token count")
        T_pad = pad_to
    token_node = np.full(T_pad, -1, np.int32)
    token_ids = np.full(T_pad, -1, np.int32)
    start = np.zeros(N, np.int32)
    end = np.zeros(N, np.int32)
    parent = np.full(N, -1, np.int32)
    pos = 0
    for r, n in enumerate(preorder):
        start[r] = pos
        for tok in n.tokens:
            token_node[pos] = r
            token_ids[pos] = tok
            pos += 1
        end[r] = pos - 1
        if n.parent is not None and n.parent is not trie.root:
            parent[r] = rank[id(n.parent)]
    # exit rank = largest rank inside the subtree.  In preorder a subtree is
    # the node followed by its descendants, so exit = rank + size - 1, with
    # subtree sizes summed from the leaves up (reverse preorder).
    size = np.ones(N, np.int64)
    for r in range(N - 1, -1, -1):
        if parent[r] != -1:
            size[parent[r]] += size[r]
    exit_rank = (np.arange(N) + size - 1).astype(np.int32)
    packed = PackedTrie(
        seq_ids=list(trie.seq_ids), n_tokens=n_tokens, T_pad=T_pad,
        token_node=token_node, token_ids=token_ids,
        node_entry=np.arange(N, dtype=np.int32), node_exit=exit_rank,
        node_parent=parent, node_start=start, node_end=end)
    for sid in trie.seq_ids:
        packed.seq_index[sid] = sequence_indices(packed, preorder, sid)
    return packed


def sequence_indices(packed: PackedTrie, preorder, sid: int) -> np.ndarray:
    """Packed token indices of sequence ``sid`` in order: the concatenation of
    the spans of the nodes it passes (``get_sequence_tree_indices``)."""
    spans = [(int(packed.node_start[r]), int(packed.node_end[r]))
             for r, n in enumerate(preorder) if sid in n.seq_ids]
    spans.sort()
    out = [np.arange(s, e + 1, dtype=np.int32) for s, e in spans]
    return np.concatenate(out) if out else np.zeros(0, np.int32)


def pack_sequences(seqs, max_tokens_per_mb: int, block: int = 128,
                   compress_nodes: bool = True, pad_to_max: bool = False):
    """Validate, pack (FFD), optionally compress, and lay out every trie."""
    if max_tokens_per_mb is None or max_tokens_per_mb <= 0:
        raise ValueError("max_tokens_per_mb must be a positive value")
    if max_tokens_per_mb % block:
        raise ValueError("max_tokens_per_mb must be a multiple of the block")
    for s in seqs:
        if len(s) == 0:
            raise ValueError("empty sequence")
        if len(s) > max_tokens_per_mb:
            raise ValueError("sequence longer than max_tokens_per_mb")
    tries = greedy_ffd(seqs, max_tokens_per_mb)
    out = []
    for t in tries:
        if compress_nodes:
            compress(t)
        out.append(layout(t, block, max_tokens_per_mb if pad_to_max else None))
    return out


def tree_token_ratio(packed_tries, seqs) -> float:
    """Metric of section "指标与监控": packed tokens / original tokens."""
    total_tree = sum(p.n_tokens for p in packed_tries)
    original = sum(len(s) for s in seqs)
    return total_tree / original

"""Oracle ancestor mask, position ids and tile classes — TEST INFRASTRUCTURE ONLY.

Definitions (AReaL Tree Training guide):

* packing figure, "注意力掩码" column: a token may attend only to tokens of
  its ancestor nodes, and causally within its own node.  Written out:
  ``M[i, j] = (j <= i) and node(j) is node(i) or an ancestor of node(i)``,
  where ancestors are found by walking parent pointers;
* section "打包数据的生成": the position id of a token is the number of tokens
  it can attend to in the dense mask, minus one;
* section "FlexAttention + BlockMask": the mask is consumed in 128x128 blocks.
  A tile with no visible pair is EMPTY, one with every pair visible is FULL,
  any other tile is PARTIAL.

Readings: a pad token (``token_node == -1``) belongs to no node, attends to
nothing and is attended by nothing; its position id is stored as 0 (the
literal "count - 1" would give -1).

Parity: pinned by the worked example of the packing figure (rows, positions,
pair count), by brute force over small tries (positions equal each token's
index within every sequence that passes it), and by the closed form
"position = depth of the token below the virtual root".
"""
from __future__ import annotations

import numpy as np

EMPTY, FULL, PARTIAL = 0, 1, 2


def ancestors_or_self(packed, node: int) -> list[int]:
    """Nodes from ``node`` up to its top-level ancestor, by parent pointers."""
    out = []
    a = node
    while a != -1:
        out.append(a)
        a = int(packed.node_parent[a])
    return out


def mask_rows(packed, r0: int, r1: int) -> np.ndarray:
    """Rows ``r0 .. r1-1`` of the dense ancestor mask, bool[r1-r0, T_pad]."""
    T = packed.T_pad
    rows = np.zeros((r1 - r0, T), dtype=bool)
    for i in range(r0, r1):
        n = int(packed.token_node[i])
        if n < 0:
            continue
        row = rows[i - r0]
        for a in ancestors_or_self(packed, n):
            row[packed.node_start[a]: packed.node_end[a] + 1] = True
        row[i + 1:] = False          # j <= i
    return rows


def ancestor_mask(packed) -> np.ndarray:
    """The dense bool mask ``[T_pad, T_pad]`` (small tries only)."""
    return mask_rows(packed, 0, packed.T_pad)


def position_ids(packed, block: int = 128) -> np.ndarray:
    """Attendable-token count minus one per row; pads get 0."""
    T = packed.T_pad
    pos = np.zeros(T, np.int32)
    for r0 in range(0, T, block):
        rows = mask_rows(packed, r0, min(T, r0 + block))
        cnt = rows.sum(axis=1)
        real = packed.token_node[r0:r0 + rows.shape[0]] >= 0
        pos[r0:r0 + rows.shape[0]] = np.where(real, cnt - 1, 0)
    return pos


def tile_classes(packed, block: int = 128) -> np.ndarray:
    """uint8[nb, nb] tile classes from the popcount of each mask tile."""
    T = packed.T_pad
    if T % block:
        raise ValueError("packed length must be a multiple of the block")
    nb = T // block
    cls = np.zeros((nb, nb), np.uint8)
    for qa in range(nb):
        rows = mask_rows(packed, qa * block, (qa + 1) * block)
        counts = rows.reshape(block, nb, block).sum(axis=(0, 2))
        cls[qa] = np.where(counts == 0, EMPTY,
                           np.where(counts == block * block, FULL, PARTIAL))
    return cls


def visible_pairs(packed) -> int:
    """Number of visible (i, j) pairs = sum over real rows of their popcount."""
    pos = position_ids(packed)
    real = packed.token_node >= 0
    return int((pos[real].astype(np.int64) + 1).sum())

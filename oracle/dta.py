"""Oracle DFS traversal schedule of dynamic tree attention — TEST INFRASTRUCTURE ONLY.

Follows "AREAL-DTA: Dynamic Tree Attention for Efficient Reinforcement
Learning of Large Language Models", sections 3.1 (depth-first traversal of
the prefix tree) and 3.2 (system optimisations), at the level of the
attention operator:

* 3.1: a stack holds the current root-to-node path, its tokens and their
  key/value states.  Descending into a node runs the forward of the node's
  new tokens against the stack's keys/values and pushes their keys/values.
  At a leaf the sequence is complete: its loss gradient is injected and the
  backward of the branch starts at once.  Popping a node runs its backward,
  by which time every descendant leaf has added its contribution to the
  gradients of the node's keys/values; the node is then dropped.
* 3.2 "chunked backward for long sequences": a path is processed in chunks
  of at most ``chunk`` tokens (2048 on the page); each chunk is a unit of
  forward, push, backward and pop.
* 3.2 "avoiding leaf KV caching": the leaf's last chunk is never pushed; its
  forward and backward run back to back.
* 3.2 "optimal DFS order": a greedy order that favours long uninterrupted
  push/pop runs.

Readings where the page is silent:
* chunks cut each node's token span from the node's first token, every
  ``chunk`` tokens (a node shorter than ``chunk`` is one chunk);
* the greedy order visits a node's children by decreasing depth in tokens
  (the longest root-to-leaf continuation below the child's first token),
  ties by preorder rank;
* at the operator level a chunk's backward needs no recomputed forward
  graph: it reads the forward's saved O and LSE (the page's recomputation
  rebuilds the layers' activations, not the attention's);
* pads belong to no node and are never scheduled.

Schedule: a list of ``(kind, t0, t1)`` over packed token rows ``[t0, t1)``
with kinds FWD_PUSH (forward of the rows against the stack, then push),
FWD_BWD (a leaf's last chunk: forward and backward, no push) and BWD_POP
(backward of the rows on top of the stack, then pop).

Parity: pinned by a hand-derived schedule of the packing figure's trie, by
structural invariants (every real token in exactly one forward and one
backward; stack discipline; the stack at a chunk's forward is exactly the
chunk's ancestor tokens in the dense mask; peak stack size), and by running
attention through the schedule: the result equals the packed tree attention
oracle (dense-mask forward and backward) for every chunk size.  See
tests/test_oracle_dta.py.
"""
from __future__ import annotations

import numpy as np

FWD_PUSH, FWD_BWD, BWD_POP = 0, 1, 2


def children(packed) -> tuple[list[list[int]], list[int]]:
    """(children of every node, top-level nodes), each list in preorder rank."""
    kids: list[list[int]] = [[] for _ in range(packed.n_nodes)]
    top: list[int] = []
    for n in sorted(range(packed.n_nodes), key=lambda n: int(packed.node_entry[n])):
        par = int(packed.node_parent[n])
        (kids[par] if par >= 0 else top).append(n)
    return kids, top


def depth_tokens(packed, kids) -> np.ndarray:
    """Tokens on the longest path from a node's first token down to a leaf."""
    depth = np.zeros(packed.n_nodes, np.int64)
    for n in sorted(range(packed.n_nodes), key=lambda n: -int(packed.node_entry[n])):
        own = int(packed.node_end[n]) - int(packed.node_start[n]) + 1
        depth[n] = own + max((depth[c] for c in kids[n]), default=0)
    return depth


def greedy_order(nodes, depth, packed) -> list[int]:
    """Deepest first, ties by preorder rank."""
    return sorted(nodes, key=lambda n: (-int(depth[n]), int(packed.node_entry[n])))


def chunks(packed, n: int, chunk: int) -> list[tuple[int, int]]:
    s, e = int(packed.node_start[n]), int(packed.node_end[n]) + 1
    return [(a, min(a + chunk, e)) for a in range(s, e, chunk)]


def schedule(packed, chunk: int = 2048):
    """The DFS traversal as a list of (kind, t0, t1)."""
    if chunk < 1:
        raise ValueError("chunk must be positive")
    kids, top = children(packed)
    depth = depth_tokens(packed, kids)
    ops: list[tuple[int, int, int]] = []

    def visit(n):
        segs = chunks(packed, n, chunk)
        leaf = not kids[n]
        pushed = segs[:-1] if leaf else segs
        for t0, t1 in pushed:
            ops.append((FWD_PUSH, t0, t1))
        if leaf:
            t0, t1 = segs[-1]
            ops.append((FWD_BWD, t0, t1))
        for c in greedy_order(kids[n], depth, packed):
            visit(c)
        for t0, t1 in reversed(pushed):
            ops.append((BWD_POP, t0, t1))

    for n in greedy_order(top, depth, packed):
        visit(n)
    return ops


def peak_stack_tokens(ops) -> int:
    cur = peak = 0
    for kind, t0, t1 in ops:
        if kind == FWD_PUSH:
            cur += t1 - t0
            peak = max(peak, cur)
        elif kind == BWD_POP:
            cur -= t1 - t0
    return peak


def run_attention(q, k, v, do, packed, chunk: int = 2048, scale=None):
    """Attention forward and backward executed through the schedule with an
    explicit key/value stack, float64.  Returns O, LSE, dQ, dK, dV in the
    packed layout (Q, O, dO, dQ ``[T, Hq, d]``; K, V, dK, dV ``[T, Hkv, d]``;
    LSE ``[Hq, T]``); pads stay zero (LSE -inf)."""
    T, Hq, d = q.shape
    g = Hq // k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    o = np.zeros_like(q)
    lse = np.full((Hq, T), -np.inf)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    stack: list[tuple[int, int]] = []

    def keys_for(t0, t1, own_pushed):
        rng = [np.arange(a, b) for a, b in stack]
        if not own_pushed:
            rng.append(np.arange(t0, t1))
        return np.concatenate(rng)

    def forward(t0, t1, keys):
        rows = np.arange(t0, t1)
        vis = keys[None, :] <= rows[:, None]          # stack keys < t0; own rows causal
        for h in range(Hq):
            kv = h // g
            s = scale * (q[rows, h, :] @ k[keys, kv, :].T)
            s = np.where(vis, s, -np.inf)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            l_ = e.sum(axis=1)
            o[rows, h, :] = (e / l_[:, None]) @ v[keys, kv, :]
            lse[h, rows] = m + np.log(l_)

    def backward(t0, t1, keys):
        rows = np.arange(t0, t1)
        vis = keys[None, :] <= rows[:, None]
        for h in range(Hq):
            kv = h // g
            s = scale * (q[rows, h, :] @ k[keys, kv, :].T)
            p = np.where(vis, np.exp(s - lse[h, rows][:, None]), 0.0)
            dv[keys, kv, :] += p.T @ do[rows, h, :]
            dp = do[rows, h, :] @ v[keys, kv, :].T
            D = (do[rows, h, :] * o[rows, h, :]).sum(axis=1)
            ds = p * (dp - D[:, None])
            dq[rows, h, :] += scale * (ds @ k[keys, kv, :])
            dk[keys, kv, :] += scale * (ds.T @ q[rows, h, :])

    for kind, t0, t1 in schedule(packed, chunk):
        if kind == FWD_PUSH:
            forward(t0, t1, keys_for(t0, t1, False))
            stack.append((t0, t1))
        elif kind == FWD_BWD:
            keys = keys_for(t0, t1, False)
            forward(t0, t1, keys)
            backward(t0, t1, keys)
        else:
            if not stack or stack[-1] != (t0, t1):
                raise AssertionError("pop does not match the stack top")
            backward(t0, t1, keys_for(t0, t1, True))
            stack.pop()
    if stack:
        raise AssertionError("stack not empty at the end")
    return o, lse, dq, dk, dv

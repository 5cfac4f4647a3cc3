"""Pins for the oracle's DFS traversal schedule of dynamic tree attention
(CPU only).

The schedule is checked against a hand-derived worked example
(tests/golden), against the dense ancestor mask (the stack at every forward
is exactly the chunk's ancestor tokens; every row that sees a chunk has run
its backward by the time the chunk is popped), against closed forms (peak
stack size), and by running attention through it: the result must equal
the packed tree attention oracle for every chunk size.
"""
import json
import os

import numpy as np
import pytest

import workloads as W
from oracle import attention as OA
from oracle import dta as OD
from oracle import mask as OM
from oracle import trie as OT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_worked_example_schedules():
    g = _golden("worked_example.json")
    gd = _golden("worked_example_dta.json")
    (p,) = OT.pack_sequences(g["sequences"], g["max_tokens_per_mb"])
    for chunk, ops in gd["schedules"].items():
        got = OD.schedule(p, int(chunk))
        assert [list(o) for o in got] == ops
        assert OD.peak_stack_tokens(got) == gd["peak_stack_tokens"][chunk]


def _random_tries(seed, n, max_len, alphabet, cap=1024):
    rng = W.SplitMix64(seed)
    out = []
    for _ in range(n):
        seqs = W.random_sequences(rng, rng.randint(1, 9), max_len, alphabet)
        out.extend(OT.pack_sequences(seqs, cap))
    return out


def _check_structure(p, chunk):
    ops = OD.schedule(p, chunk)
    M = OM.ancestor_mask(p)
    real = np.nonzero(p.token_node >= 0)[0]
    fwd = np.zeros(p.T_pad, int)
    bwd = np.zeros(p.T_pad, int)
    bwd_at = np.full(p.T_pad, -1)
    stack = []
    for idx, (kind, t0, t1) in enumerate(ops):
        assert 0 < t1 - t0 <= chunk
        assert len({int(p.token_node[i]) for i in range(t0, t1)}) == 1   # inside one node
        if kind in (OD.FWD_PUSH, OD.FWD_BWD):
            fwd[t0:t1] += 1
            on_stack = sorted(i for a, b in stack for i in range(a, b))
            assert on_stack == np.nonzero(M[t0, :t0])[0].tolist()       # exactly the ancestors
        if kind == OD.FWD_PUSH:
            stack.append((t0, t1))
        if kind in (OD.FWD_BWD, OD.BWD_POP):
            bwd[t0:t1] += 1
            bwd_at[t0:t1] = idx
        if kind == OD.BWD_POP:
            assert stack and stack[-1] == (t0, t1)
            stack.pop()
        if kind == OD.FWD_BWD:
            node = int(p.token_node[t0])
            assert t1 == p.node_end[node] + 1                             # a leaf's last chunk
            assert not (p.node_parent == node).any()
    assert not stack
    assert (fwd[real] == 1).all() and (bwd[real] == 1).all()
    assert (fwd[p.token_node < 0] == 0).all()
    # a token's backward comes after (or with) the backward of every row that sees it
    for j in real:
        rows = np.nonzero(M[:, j])[0]
        assert (bwd_at[rows] <= bwd_at[j]).all()
    # closed form: the peak is the longest root-to-leaf path minus its leaf's last chunk
    kids, _ = OD.children(p)
    best = 0
    for n in range(p.n_nodes):
        if kids[n]:
            continue
        path = int(np.count_nonzero(M[int(p.node_end[n])]))
        last = (int(p.node_end[n]) - int(p.node_start[n])) % chunk + 1
        best = max(best, path - last)
    assert OD.peak_stack_tokens(ops) == best
    return ops


@pytest.mark.parametrize("chunk", [1, 2, 5, 64, 2048])
def test_structure_random_tries(chunk):
    for p in _random_tries(100 + chunk, 12, 40, 3):
        _check_structure(p, chunk)


def test_greedy_order_deepest_child_first():
    for p in _random_tries(7, 10, 30, 2):
        kids, top = OD.children(p)
        depth = OD.depth_tokens(p, kids)
        ops = OD.schedule(p, 4096)
        first_fwd = {}
        for idx, (kind, t0, _) in enumerate(ops):
            if kind != OD.BWD_POP:
                first_fwd.setdefault(int(p.token_node[t0]), idx)
        for group in kids + [top]:
            order = sorted(group, key=lambda n: first_fwd[n])
            ds = [int(depth[n]) for n in order]
            assert ds == sorted(ds, reverse=True)
        # the depth is the longest path below the node's first token, by brute force
        M = OM.ancestor_mask(p)
        for n in range(p.n_nodes):
            s = int(p.node_start[n])
            below = [i for i in range(p.T_pad) if M[i, s]]
            longest = max(int(np.count_nonzero(M[i, s:])) for i in below)
            assert depth[n] == longest


@pytest.mark.parametrize("chunk,g", [(1, 1), (3, 2), (64, 1), (2048, 2)])
def test_attention_through_the_schedule_equals_tree_attention(chunk, g):
    rng = W.SplitMix64(900 + chunk)
    seqs = W.random_sequences(rng, 6, 50, 2)
    (p,) = OT.pack_sequences(seqs, 1024)
    Hkv, d = 2, 16
    t = W.tensors(p.T_pad, Hkv * g, Hkv, d, seed=chunk)
    q, k, v, do = (t[n].float().numpy().astype(np.float64) for n in ("q", "k", "v", "do"))
    M = OM.ancestor_mask(p)
    o_ref, lse_ref = OA.forward(q, k, v, M)
    dq_ref, dk_ref, dv_ref = OA.backward(q, k, v, o_ref, do, M)
    o, lse, dq, dk, dv = OD.run_attention(q, k, v, do, p, chunk)
    real = p.token_node >= 0
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[:, real], lse_ref[:, real], rtol=0, atol=1e-12)
    assert np.isneginf(lse[:, ~real]).all()
    for got, want in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-11)


def test_chunk_must_be_positive():
    (p,) = OT.pack_sequences([[1, 2]], 128)
    with pytest.raises(ValueError):
        OD.schedule(p, 0)
